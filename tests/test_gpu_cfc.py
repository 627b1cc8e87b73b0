"""CfC K-loop forward + backward on the GPU, through the C ABI, against the
oracle, on the benchmark workloads (full size) and on ragged edge cases."""

import numpy as np
import pytest

import oracle
import recurrent_cell_gb300 as cfc
from recurrent_cell_gb300 import workloads as wl
from gpu_common import PARITY_BIAS, CfcRun, assert_close, dev, require_gpu, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def oracle_ref(w, inp, per_sample=True, **seeds):
    return oracle.backward(inp["x"], inp["h0"], inp["W_in"], inp["W_rec"], inp["b"], inp["dt"],
                           mode=w.math, per_sample=per_sample, **seeds)


def check_all(w, got, ref, keys=("h_seq", "grad_W_in", "grad_W_rec", "grad_b", "grad_h0", "grad_x")):
    for k in keys:
        assert_close(got[k], ref[k], w.math, f"{w.name}:{k}",
                     state_bf16=(k == "h_seq" and w.math == wl.MATH_BF16))


def run(w, inp, grad_path=None, **bw):
    r = CfcRun(w, inp, grad_path=grad_path)
    r.forward()
    r.backward(**bw)
    return r, r.results()


# ------------------------------------------------------------- benchmark workloads

def test_tiny_fp32_all_upstream_seeds():
    w = wl.TINY
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    rng = np.random.default_rng(1)
    gseq = rng.standard_normal((w.B, w.K, w.n_hid)).astype(np.float32)
    glast = rng.standard_normal((w.B, w.n_hid)).astype(np.float32)
    r, got = run(w, inp, y=True, grad_h_seq=dev(gseq), grad_h_last=dev(glast))
    ref = oracle_ref(w, inp, y=inp["y"], grad_h_seq=gseq, grad_h_last=glast)
    check_all(w, got, ref)
    assert_close(got["per_sample"], ref["per_sample"], w.math, "tiny:per_sample")


SEEDS = [
    wl.Workload("seeds_tf32_B70_K4_H160", B=70, K=4, n_in=24, n_hid=160, math=wl.MATH_TF32),
    wl.Workload("seeds_bf16_B37_K5_H40", B=37, K=5, n_in=24, n_hid=40, math=wl.MATH_BF16,
                dt_per_sample=True),
]


@pytest.mark.parametrize("kernels", ["auto", "tc", "tcs", "cluster", "simt", "solo", "solo16"])
@pytest.mark.parametrize("w", SEEDS, ids=lambda w: w.name)
def test_upstream_seeds_every_family(w, kernels, monkeypatch):
    """Per-step seeds grad_h_seq, the last state's grad_h_last and the y
    loss together, through every K-loop family of the reduced-precision
    modes (each loads the per-step seeds in its own way)."""
    set_kernels(monkeypatch, kernels)
    inp = wl.make_inputs(w, seed=17, bias_scale=PARITY_BIAS)
    rng = np.random.default_rng(2)
    gseq = rng.standard_normal((w.B, w.K, w.n_hid)).astype(np.float32)
    glast = rng.standard_normal((w.B, w.n_hid)).astype(np.float32)
    r, got = run(w, inp, y=True, grad_h_seq=dev(gseq), grad_h_last=dev(glast))
    ref = oracle_ref(w, inp, y=inp["y"], grad_h_seq=gseq, grad_h_last=glast)
    check_all(w, got, ref)
    assert_close(got["per_sample"], ref["per_sample"], w.math, f"{w.name}:per_sample")


def test_smoke_fp32_scratch_path():
    w = wl.SMOKE
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    r, got = run(w, inp)
    ref = oracle_ref(w, inp, y=inp["y"])
    check_all(w, got, ref)
    assert_close(got["per_sample"], ref["per_sample"], w.math, "smoke:per_sample")


def set_kernels(monkeypatch, kernels):
    """Kernel family for the K loops; "solo16" is the single-block family
    with 16-sample blocks (8 a thread) instead of the automatic tile."""
    if kernels == "solo16":
        monkeypatch.setenv("CFC_KLOOP_KERNELS", "solo")
        monkeypatch.setenv("CFC_SOLO_TILE", "16")
    else:
        monkeypatch.setenv("CFC_KLOOP_KERNELS", kernels)
        monkeypatch.delenv("CFC_SOLO_TILE", raising=False)


@pytest.mark.parametrize("kernels", ["tc", "tcs", "cluster", "simt", "solo", "solo16"])
@pytest.mark.parametrize("w", [wl.TINY, wl.SMOKE, wl.MID.with_(B=128, K=16),
                               wl.LARGE.with_(B=96, K=4)], ids=lambda w: w.name)
def test_kernel_families_on_benchmark_shapes(w, kernels, monkeypatch):
    set_kernels(monkeypatch, kernels)
    inp = wl.make_inputs(w, seed=9, bias_scale=PARITY_BIAS)
    r, got = run(w, inp)
    ref = oracle_ref(w, inp, per_sample=False, y=inp["y"])
    check_all(w, got, ref)


@pytest.mark.parametrize("variant", ["tma", "staged"])
@pytest.mark.parametrize("base", [wl.LARGE.with_(B=512), wl.MID.with_(B=96, K=32)],
                         ids=lambda w: w.name.split("_")[0])
def test_weight_gradient_contractions(base, variant, monkeypatch):
    """The TMA-fed weight-gradient contraction and the register-staged one,
    on the large (bf16) and mid (TF32) shapes with fewer samples."""
    if variant == "staged":
        monkeypatch.setenv("CFC_WGRAD_STAGED", "1")
    w = base
    inp = wl.make_inputs(w, seed=21, bias_scale=PARITY_BIAS)
    r, got = run(w, inp)
    ref = oracle_ref(w, inp, per_sample=False, y=inp["y"])
    check_all(w, got, ref)


def test_smoke_fp32_gemm_path_matches():
    w = wl.SMOKE
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    r, got = run(w, inp, grad_path=wl.GRAD_GEMM)
    ref = oracle_ref(w, inp, per_sample=False, y=inp["y"])
    check_all(w, got, ref)


def test_mid_tf32_full_size():
    w = wl.MID
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    r, got = run(w, inp)
    ref = oracle_ref(w, inp, per_sample=False, y=inp["y"])
    check_all(w, got, ref)


def test_large_bf16_full_size():
    w = wl.LARGE
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    r, got = run(w, inp)
    ref = oracle_ref(w, inp, per_sample=False, y=inp["y"])
    check_all(w, got, ref)


# ------------------------------------------------------------- ragged / edge shapes

EDGE = [
    wl.Workload("edge_B1_K1", B=1, K=1, n_in=3, n_hid=5),
    wl.Workload("edge_B701_K3_odd", B=701, K=3, n_in=7, n_hid=33),            # BT=4, ragged tail
    wl.Workload("edge_B5_K6_tf32", B=5, K=6, n_in=24, n_hid=48, math=wl.MATH_TF32),
    wl.Workload("edge_B37_K5_bf16", B=37, K=5, n_in=24, n_hid=40, math=wl.MATH_BF16,
                dt_per_sample=True),
    wl.Workload("edge_B3000_K2_bf16", B=3000, K=2, n_in=40, n_hid=72, math=wl.MATH_BF16,
                grad_path=wl.GRAD_GEMM, dt_per_sample=True),
    wl.Workload("edge_wide_H600", B=3, K=2, n_in=100, n_hid=600),            # units loop (>512 threads)
    # staged grad_x after the cluster backward: 35 rows (a ragged 32-row tile)
    # and 68 input columns (a second, 4-wide column block)
    wl.Workload("edge_gx_B7_K5_n68", B=7, K=5, n_in=68, n_hid=44, dt_per_sample=True),
    # tensor-core K loop: cluster of H/32 blocks, ragged batch tiles, K padding
    wl.Workload("edge_tc_tf32_B70_K3", B=70, K=3, n_in=16, n_hid=64, math=wl.MATH_TF32),
    wl.Workload("edge_tc_bf16_B45_K5", B=45, K=5, n_in=40, n_hid=96, math=wl.MATH_BF16,
                dt_per_sample=True),
    wl.Workload("edge_tc_bf16_odd_n_in", B=19, K=4, n_in=7, n_hid=32, math=wl.MATH_BF16),
    # streamed-weight K loops with two unit halves: H0 = 128 not on an atom
    # pair boundary, x / h atoms shared, a short second half
    wl.Workload("edge_tcs_bf16_H200", B=150, K=3, n_in=40, n_hid=200, math=wl.MATH_BF16,
                dt_per_sample=True),
    wl.Workload("edge_tcs_tf32_H160", B=70, K=4, n_in=24, n_hid=160, math=wl.MATH_TF32),
    # three and four unit blocks: a second half of two blocks, longer schedules
    wl.Workload("edge_tcs_bf16_H384", B=70, K=3, n_in=64, n_hid=384, math=wl.MATH_BF16,
                dt_per_sample=True),
    wl.Workload("edge_tcs_bf16_H512", B=40, K=2, n_in=64, n_hid=512, math=wl.MATH_BF16),
    # single-block tensor-core kernels: ragged last tile (B = 37), n_hid not a
    # multiple of 32 (idle TMEM lanes) and n_hid = 128 exactly in bf16
    wl.Workload("edge_solo_tf32_B37_H100", B=37, K=4, n_in=20, n_hid=100, math=wl.MATH_TF32,
                dt_per_sample=True),
    wl.Workload("edge_solo_bf16_B20_H128", B=20, K=6, n_in=64, n_hid=128, math=wl.MATH_BF16),
    # rows that are not 16-byte aligned (n_hid % 4, n_in odd): the single-block
    # kernels' element-wise weight staging
    wl.Workload("edge_solo_tf32_H66_odd_n_in", B=19, K=5, n_in=13, n_hid=66, math=wl.MATH_TF32,
                dt_per_sample=True),

    # TMA-fed weight gradient (bf16, GEMM path): 64 steps of one sample per
    # chunk with a ragged 3H tile, and whole samples per chunk
    wl.Workload("edge_tma_K128_H64", B=3, K=128, n_in=64, n_hid=64, math=wl.MATH_BF16,
                grad_path=wl.GRAD_GEMM),
    wl.Workload("edge_tma_B40_K8", B=40, K=8, n_in=64, n_hid=128, math=wl.MATH_BF16,
                grad_path=wl.GRAD_GEMM, dt_per_sample=True),
    # the same in TF32 (32-row chunks, rounding warps): whole samples per chunk
    # with a ragged 3H tile, and 32 steps of one sample per chunk
    wl.Workload("edge_tma_tf32_B40_K8", B=40, K=8, n_in=32, n_hid=64, math=wl.MATH_TF32,
                grad_path=wl.GRAD_GEMM, dt_per_sample=True),
    wl.Workload("edge_tma_tf32_K64_H32", B=3, K=64, n_in=32, n_hid=32, math=wl.MATH_TF32,
                grad_path=wl.GRAD_GEMM),
    # two samples per 32-row chunk, three x boxes
    wl.Workload("edge_tma_tf32_K16_n96", B=20, K=16, n_in=96, n_hid=64, math=wl.MATH_TF32,
                grad_path=wl.GRAD_GEMM, dt_per_sample=True),
]


# One and two steps through the single-block kernels (the automatic choice
# takes them for these shapes): the look-ahead input part and the x staging
# stop early, the backward's first step is also its last.
EDGE_SHORT = [
    wl.Workload("edge_solo_tf32_K1", B=21, K=1, n_in=64, n_hid=128, math=wl.MATH_TF32),
    wl.Workload("edge_solo_bf16_K2", B=9, K=2, n_in=32, n_hid=64, math=wl.MATH_BF16, dt_per_sample=True),
]


@pytest.mark.parametrize("kernels", ["auto", "solo", "solo16"])
@pytest.mark.parametrize("w", EDGE_SHORT, ids=lambda w: w.name)
@pytest.mark.parametrize("path", [wl.GRAD_SCRATCH, wl.GRAD_GEMM])
def test_short_loops_single_block(w, path, kernels, monkeypatch):
    set_kernels(monkeypatch, kernels)
    inp = wl.make_inputs(w, seed=5, bias_scale=PARITY_BIAS)
    r, got = run(w, inp, grad_path=path)
    ref = oracle_ref(w, inp, per_sample=(path == wl.GRAD_SCRATCH), y=inp["y"])
    check_all(w, got, ref)
    if path == wl.GRAD_SCRATCH:
        assert_close(got["per_sample"], ref["per_sample"], w.math, f"{w.name}:per_sample")


@pytest.mark.parametrize("kernels", ["auto", "tc", "tcs", "cluster", "simt", "solo", "solo16"])
@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
@pytest.mark.parametrize("path", [wl.GRAD_SCRATCH, wl.GRAD_GEMM])
def test_edge_shapes(w, path, kernels, monkeypatch):
    """Both K-loop kernel families (cluster-resident weights, streaming
    weights) and the automatic choice, on ragged shapes."""
    set_kernels(monkeypatch, kernels)
    inp = wl.make_inputs(w, seed=5, bias_scale=PARITY_BIAS)
    r, got = run(w, inp, grad_path=path)
    ref = oracle_ref(w, inp, per_sample=(path == wl.GRAD_SCRATCH), y=inp["y"])
    check_all(w, got, ref)
    if path == wl.GRAD_SCRATCH:
        assert_close(got["per_sample"], ref["per_sample"], w.math, f"{w.name}:per_sample")


# ------------------------------------------------------------- invariants

def test_run_to_run_bit_identical():
    for w in (wl.SMOKE, wl.MID.with_(B=256, K=16)):
        inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
        r = CfcRun(w, inp)
        first = None
        for _ in range(10 if w is wl.SMOKE else 3):
            r.forward()
            r.backward()
            cur = r.raw()
            if first is None:
                first = cur
            else:
                for a, b in zip(first, cur):
                    np.testing.assert_array_equal(a, b)


def test_scratch_and_workspace_cleared_between_calls():
    """Call A then call B on the same buffers: B's outputs are bit-identical to
    a fresh run of B (nothing of A survives in the scratch or the workspace)."""
    w = wl.SMOKE
    inp_a = wl.make_inputs(w, seed=100, bias_scale=PARITY_BIAS)
    inp_b = wl.make_inputs(w, seed=200, bias_scale=PARITY_BIAS)
    r = CfcRun(w, inp_a)
    r.forward(); r.backward()
    r.set_inputs(inp_b)
    r.forward(); r.backward()
    reused = r.raw()
    fresh = CfcRun(w, inp_b)
    fresh.forward(); fresh.backward()
    for a, b in zip(reused, fresh.raw()):
        np.testing.assert_array_equal(a, b)


def test_single_sample_equals_its_batch_row():
    """B = 1 runs of single samples reproduce the rows of the batched run."""
    w = wl.SMOKE
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    _, full = run(w, inp)
    for i in (0, 13, 31):
        one = {k: (v[i:i + 1] if k in ("x", "h0", "y") else v) for k, v in inp.items()}
        w1 = w.with_(B=1)
        _, got = run(w1, one)
        for k in ("h_seq", "grad_h0", "grad_x", "per_sample"):
            np.testing.assert_array_equal(got[k][0], full[k][i], err_msg=k)


def test_batch_permutation_permutes_rows():
    w = wl.MID.with_(B=64, K=8)
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    perm = np.random.default_rng(3).permutation(w.B)
    pin = {k: (v[perm] if k in ("x", "h0", "y") else v) for k, v in inp.items()}
    _, a = run(w, inp)
    _, b = run(w, pin)
    for k in ("h_seq", "grad_h0", "grad_x"):
        np.testing.assert_array_equal(b[k], a[k][perm], err_msg=k)
    for k in ("grad_W_in", "grad_W_rec", "grad_b"):
        assert_close(b[k], a[k], w.math, k)


def test_optional_outputs_may_be_null():
    w = wl.TINY
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    _, full = run(w, inp)
    r = CfcRun(w, inp)
    r.forward()
    r.backward(grad_x=False, grad_h0=False)
    got = r.results()
    for k in ("grad_W_in", "grad_W_rec", "grad_b", "per_sample", "h_seq"):
        np.testing.assert_array_equal(got[k], full[k], err_msg=k)


def test_scratch_rows_reduce_to_the_gradients():
    """The scratch path's reduced gradients are reduce_axis0 of its own
    per-sample rows (the standalone entry point gives the same bits)."""
    torch = torch_mod()
    w = wl.SMOKE
    r, got = run(w, wl.make_inputs(w, bias_scale=PARITY_BIAS))
    out = torch.empty(w.N, device="cuda")
    cfc.reduce_axis0(r.scratch, out)
    packed = torch.cat([r.gWi.reshape(-1), r.gWr.reshape(-1), r.gb.reshape(-1)])
    assert torch.equal(out.view(torch.int32), packed.view(torch.int32))


def test_outputs_stay_inside_their_buffers():
    """Guard canaries: every output is a slice of a larger NaN-filled buffer;
    nothing outside the slice may change."""
    torch = torch_mod()
    w = wl.Workload("guard", B=9, K=4, n_in=12, n_hid=20)
    inp = wl.make_inputs(w, bias_scale=PARITY_BIAS)
    r = CfcRun(w, inp)
    G = 64
    bufs = {}
    for name in ("h_seq", "gWi", "gWr", "gb", "gh0", "gx", "scratch"):
        t = getattr(r, name)
        big = torch.full((t.numel() + 2 * G,), float("nan"), dtype=t.dtype, device="cuda")
        setattr(r, name, big[G:G + t.numel()].view(t.shape))
        bufs[name] = big
    r.forward()
    r.backward()
    torch.cuda.synchronize()
    for name, big in bufs.items():
        h = big.float().cpu().numpy()
        assert np.all(np.isnan(h[:G])) and np.all(np.isnan(h[-G:])), f"{name} guard overwritten"
    ref = oracle_ref(w, inp, y=inp["y"])
    check_all(w, r.results(), ref)
