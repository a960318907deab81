"""GPU MoE steps either side of the grouped GEMM vs the CPU oracle.

fp8_quantize_gathered (the routed tokens laid out in expert order and
quantised row-wise) must match the oracle's codes and scales bit for bit.
fp8_swiglu_quantize (SwiGLU of the gate+up output, quantised row-wise for the
down projection) is compared with the definition y = BF16(silu(g) * up),
evaluated in float64 and rounded once: bit for bit in every quantisation
group whose elements all lie more than 8 float32 ulps from a BF16 rounding
boundary, and, in the few groups that hold such an element, with either
admissible BF16 value accepted for it (oracle.moe.swiglu_check).  The
fraction of such elements is asserted to be small.  Cases: ragged groups,
strided rows, repeated and out-of-range token indices, every finite BF16 gate
value (e^-g overflowing float32 included), the MoE layer's full sizes
(sampled rows), and the whole layer chained through the grouped GEMMs with
each step fed the GPU's own previous output.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import gemm as OG
from oracle import moe as OM
from tests._util import assert_gemm_close, bf16_to_f64, np_f32, np_u8, to_dev_bf16, to_f32

pytestmark = pytest.mark.gpu

fp = pytest.importorskip("fp8_block_scaled_03_gb300")

GRANS = ("1x128", "mxfp8", "1x128_pow2")


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()
    assert torch.cuda.is_available()


def scales_np(s, gran):
    return np_f32(s) if gran == "1x128" else np_u8(s)


def assert_swiglu(q, s, h, inter, gran, what, max_tie_frac=1e-3):
    """GPU SwiGLU codes and scales against the float64 definition (ties aware)."""
    gs = np_f32(s) if gran == "1x128" else np_u8(s)
    mism, ties, tie_groups = OM.swiglu_check(np_u8(q), gs, h, inter, gran)
    assert mism == 0, f"{what}: {mism} code/scale entries differ ({ties} near-boundary elements)"
    assert ties <= max_tie_frac * h.shape[0] * inter + 2, f"{what}: {ties} near-boundary elements"
    return ties, tie_groups


def assert_same(q, s, pq, ps, gran, what):
    gq, gs = np_u8(q), scales_np(s, gran)
    assert gq.shape == pq.shape and gs.shape == ps.shape, what
    assert np.array_equal(gq, pq), f"{what}: {(gq != pq).sum()} code bytes differ"
    if gran == "1x128":
        assert np.array_equal(gs.view(np.uint32), ps.astype(np.float32).view(np.uint32)), f"{what}: scales differ"
    else:
        assert np.array_equal(gs, ps), f"{what}: {(gs != ps).sum()} scale bytes differ"


# ---------------------------------------------------------------- gather + quantise
@pytest.mark.parametrize("gran", GRANS)
def test_gathered_ragged_with_repeats(gran):
    tokens, cols = 301, 1000                       # 1000 = 7x128 + 104 = 31x32 + 8: ragged last groups
    bits = synth.activations((tokens, cols), seed=71, outlier_frac=0.01, outlier_mult=60.0)
    g = synth.rng(72)
    idx = g.integers(0, tokens, size=777).astype(np.int64)
    idx[:3] = [0, tokens - 1, 0]
    q, s = fp.fp8_quantize_gathered(to_dev_bf16(bits), torch.from_numpy(idx).cuda(), gran)
    torch.cuda.synchronize()
    pq, ps = OM.quantize_gathered(to_f32(bits), idx, gran)
    assert_same(q, s, pq, ps, gran, f"gathered {gran}")


@pytest.mark.parametrize("gran", GRANS)
def test_gathered_strided_rows(gran):
    tokens, cols, ld = 64, 384, 520
    full = synth.activations((tokens, ld), seed=73)
    xd = to_dev_bf16(full)[:, :cols]
    idx = np.arange(tokens - 1, -1, -1, dtype=np.int64).repeat(3)
    q, s = fp.fp8_quantize_gathered(xd, torch.from_numpy(idx).cuda(), gran)
    torch.cuda.synchronize()
    pq, ps = OM.quantize_gathered(to_f32(full[:, :cols]), idx, gran)
    assert_same(q, s, pq, ps, gran, f"gathered strided {gran}")


@pytest.mark.parametrize("gran", GRANS)
def test_gathered_out_of_range_index_zeroes_row_and_sets_status(gran):
    tokens, cols = 40, 256
    bits = synth.activations((tokens, cols), seed=74)
    idx = np.array([5, -1, 39, 40, 7, 2**40, 0], np.int64)
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    q, s = fp.fp8_quantize_gathered(to_dev_bf16(bits), torch.from_numpy(idx).cuda(), gran, ws=ws)
    assert fp.read_status(ws) == fp.EINDEX
    ok = np.array([0, 2, 4, 6])
    pq, ps = OM.quantize_gathered(to_f32(bits), idx[ok], gran)
    zq, zs = OM.ROWWISE[gran](np.zeros((1, cols), np.float32))
    gq, gs = np_u8(q), scales_np(s, gran)
    assert np.array_equal(gq[ok], pq) and np.array_equal(gs[ok], ps)
    for r in (1, 3, 5):
        assert np.array_equal(gq[r], zq[0]) and np.array_equal(gs[r], zs[0])
    fp.clear_status(ws)
    assert fp.read_status(ws) == 0
    # valid indices leave the status word alone
    fp.fp8_quantize_gathered(to_dev_bf16(bits), torch.from_numpy(idx[ok]).cuda(), gran, ws=ws)
    assert fp.read_status(ws) == 0


def test_gathered_empty_and_no_tokens():
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    q, s = fp.fp8_quantize_gathered(x, torch.zeros(0, dtype=torch.int64, device="cuda"), "mxfp8")
    assert q.shape == (0, 128)
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    q, s = fp.fp8_quantize_gathered(x, torch.zeros(4, dtype=torch.int64, device="cuda"), "mxfp8", ws=ws)
    assert fp.read_status(ws) == fp.EINDEX          # no token exists: every row is out of range
    assert int(q.count_nonzero()) == 0 and int(s.count_nonzero()) == 0


# ---------------------------------------------------------------- gather of quantised rows
@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("cols", (1000, 264, 2048))
def test_gather_rows_after_quantise_matches_oracle(gran, cols):
    """fp8_quantize of the token matrix, then fp8_gather_rows, against the
    oracle's gathered quantisation: ragged last groups and 8-byte code
    chunks (1000, 264 columns), 16-byte chunks (2048), repeated indices."""
    tokens = 301
    bits = synth.activations((tokens, cols), seed=81 + cols, outlier_frac=0.01, outlier_mult=60.0)
    idx = synth.rng(82).integers(0, tokens, size=777).astype(np.int64)
    idx[:3] = [0, tokens - 1, 0]
    qt, st, _ = fp.fp8_quantize(to_dev_bf16(bits), gran)
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    q, s = fp.fp8_gather_rows(qt, st, torch.from_numpy(idx).cuda(), gran, ws=ws)
    torch.cuda.synchronize()
    pq, ps = OM.quantize_gathered(to_f32(bits), idx, gran)
    assert_same(q, s, pq, ps, gran, "gather of quantised rows")
    assert fp.read_status(ws) == 0


@pytest.mark.parametrize("gran", GRANS)
def test_gather_rows_out_of_range_like_gathered_quantise(gran):
    """Out-of-range indices: the same all-zero rows and status as the
    gathered quantiser; no tokens at all; no rows."""
    tokens, cols = 40, 256
    bits = synth.activations((tokens, cols), seed=74)
    idx = torch.tensor([5, -1, 39, 40, 7, 2**40, 0], dtype=torch.int64, device="cuda")
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    qt, st, _ = fp.fp8_quantize(to_dev_bf16(bits), gran)
    q, s = fp.fp8_gather_rows(qt, st, idx, gran, ws=ws)
    assert fp.read_status(ws) == fp.EINDEX
    q2, s2 = fp.fp8_quantize_gathered(to_dev_bf16(bits), idx, gran, ws=ws)
    assert torch.equal(q, q2) and torch.equal(s.view(torch.uint8), s2.view(torch.uint8))
    fp.clear_status(ws)
    none_q = torch.zeros((0, cols), dtype=torch.uint8, device="cuda")
    shp, dt = fp.scale_shape(gran, 0, cols)
    none_s = torch.zeros(shp, dtype=dt, device="cuda")
    q, s = fp.fp8_gather_rows(none_q, none_s, idx[:4], gran, ws=ws)
    assert fp.read_status(ws) == fp.EINDEX           # no token exists: every row is out of range
    zq, zs = OM.ROWWISE[gran](np.zeros((1, cols), np.float32))
    assert np.array_equal(np_u8(q), np.repeat(zq, 4, axis=0))
    assert np.array_equal(scales_np(s, gran), np.repeat(zs, 4, axis=0))
    q, s = fp.fp8_gather_rows(qt, st, torch.zeros(0, dtype=torch.int64, device="cuda"), gran)
    assert q.shape == (0, cols)


@pytest.mark.parametrize("gran", ("mxfp8", "1x128"))
def test_gather_rows_full_moe_layer_equals_gathered_quantise(gran):
    """MoE layer size (16384 tokens x 2048, top-8 of 128 experts): the two
    paths give the same bytes, compared on the device in full."""
    tokens, hidden, experts, topk = 16384, 2048, 128, 8
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = (torch.randn((tokens, hidden), generator=g, device="cuda")).to(torch.bfloat16)
    order, _ = synth.moe_routing(tokens, experts, topk, seed=0)
    idx = torch.from_numpy(np.asarray(order, dtype=np.int64)).cuda()
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    qt, st, _ = fp.fp8_quantize(x, gran, ws=ws)
    q, s = fp.fp8_gather_rows(qt, st, idx, gran, ws=ws)
    q2, s2 = fp.fp8_quantize_gathered(x, idx, gran, ws=ws)
    assert torch.equal(q, q2) and torch.equal(s.view(torch.uint8), s2.view(torch.uint8))
    assert fp.read_status(ws) == 0


@pytest.mark.parametrize("gran", ("mxfp8", "1x128"))
def test_gathered_full_moe_layer_sampled(gran):
    """Routed tokens of the MoE layer (16384 tokens x 2048, 128 experts, top 8:
    131072 rows): every row checked for 256 sampled rows, and the scales of
    all rows against the per-token oracle quantisation of x."""
    tokens, hidden = 16384, 2048
    bits = synth.activations((tokens, hidden), seed=75, outlier_frac=0.001, outlier_mult=100.0)
    idx, _ = synth.moe_routing(tokens, 128, 8, seed=0)
    q, s = fp.fp8_quantize_gathered(to_dev_bf16(bits), torch.from_numpy(idx).cuda(), gran)
    torch.cuda.synchronize()
    rows = synth.rng(76).choice(idx.size, 256, replace=False)
    rows[:2] = [0, idx.size - 1]
    pq, ps = OM.quantize_gathered(to_f32(bits), idx[rows], gran)
    gq, gs = np_u8(q[torch.from_numpy(rows).cuda()]), scales_np(s[torch.from_numpy(rows).cuda()], gran)
    assert np.array_equal(gq, pq) and np.array_equal(gs, ps)
    # property at any size: row r of the gathered result is row idx[r] of the per-token quantisation
    qt, st, _ = fp.fp8_quantize(to_dev_bf16(bits), gran)
    it = torch.from_numpy(idx).cuda()
    assert torch.equal(q, qt[it]) and torch.equal(s, st[it])


# ---------------------------------------------------------------- SwiGLU + requantise
@pytest.mark.parametrize("gran", GRANS)
def test_swiglu_ragged(gran):
    rows, inter = 333, 776                          # 776 = 6x128 + 8 = 24x32 + 8
    bits = synth.activations((rows, 2 * inter), seed=81, outlier_frac=0.02, outlier_mult=30.0)
    q, s = fp.fp8_swiglu_quantize(to_dev_bf16(bits), gran)
    torch.cuda.synchronize()
    assert_swiglu(q, s, to_f32(bits), inter, gran, f"swiglu {gran}")


@pytest.mark.parametrize("gran", GRANS)
def test_swiglu_strided_and_wider_rows(gran):
    rows, inter, ld = 96, 256, 640                  # h rows hold more than [gate | up]
    full = synth.activations((rows, ld), seed=82)
    hd = to_dev_bf16(full)[:, :ld - 64]
    q, s = fp.fp8_swiglu_quantize(hd, gran, inter)
    torch.cuda.synchronize()
    assert_swiglu(q, s, to_f32(full), inter, gran, f"swiglu strided {gran}")


def all_finite_bf16():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    e = (b >> 7) & 0xFF
    return b[e != 0xFF]


@pytest.mark.parametrize("upv", (1.0, -0.75))
def test_swiglu_every_bf16_gate_value_exact_y(upv):
    """Every finite BF16 gate value (so e^-g runs over its whole range,
    beyond float32 overflow included), each alone in its 1x128 group: the
    group's FP32 scale is |y| / 448 rounded once, which fixes |y| (distinct
    BF16 values give distinct quotients), and the code fixes the sign, so y
    itself is compared with the definition."""
    g = all_finite_bf16()
    per_row = 64
    inter = 128 * per_row
    rows = -(-g.size // per_row)
    gate = np.zeros((rows * per_row, 128), np.uint16)
    gate[:g.size, 0] = g
    gate = gate.reshape(rows, inter)
    up = np.full((rows, inter), synth.f32_to_bf16_bits(np.array([upv], np.float32))[0], np.uint16)
    h = np.concatenate([gate, up], axis=1)
    q, s = fp.fp8_swiglu_quantize(to_dev_bf16(h), "1x128")
    torch.cuda.synchronize()
    # up = -0.75 puts many y exactly at BF16 midpoints give or take a hair:
    # silu(g) * 0.75 is a 10-bit product of 8-bit values where silu(g) is
    # g / 2 (tiny g) or g (large g), so a quarter of those land within the
    # band by construction (21 % of all gates; 0.4 % with up = 1)
    assert_swiglu(q, s, to_f32(h), inter, "1x128", f"swiglu single gates up={upv}", max_tie_frac=0.25)


@pytest.mark.parametrize("gran", GRANS)
def test_swiglu_every_bf16_gate_value_mixed_groups(gran):
    """Every finite BF16 gate value, shuffled so groups mix magnitudes,
    against several up values."""
    g = all_finite_bf16()
    inter = 1024
    n = g.size
    rows = -(-n // inter)
    gate = np.zeros(rows * inter, np.uint16)
    gate[:n] = synth.rng(83).permutation(g)
    gate = gate.reshape(rows, inter)
    for upv in (1.0, -0.75, 0.0078125):              # |up| <= 1 keeps silu(g) * up finite
        up = np.full((rows, inter), synth.f32_to_bf16_bits(np.array([upv], np.float32))[0], np.uint16)
        h = np.concatenate([gate, up], axis=1)
        q, s = fp.fp8_swiglu_quantize(to_dev_bf16(h), gran)
        torch.cuda.synchronize()
        # as in the single-gate test: up = -0.75 puts 21 % of the elements in the band
        assert_swiglu(q, s, to_f32(h), inter, gran, f"swiglu all gates up={upv} {gran}", max_tie_frac=0.25)


def test_swiglu_isolated_values_exact():
    """Special gate values (0, +-1, +-20, either side of the e^x overflow and
    underflow thresholds, tiny and large), each alone in its 32-element
    group."""
    inter = 32 * 64
    vals = np.array([0.0, 1.0, -1.0, 20.0, -20.0, 88.0, -88.0, 90.0, -90.0, 0.5, -0.5, 3.0e-5, -3.0e-5,
                     100.0, -100.0, 7.25], np.float32)
    gate = np.zeros((1, inter), np.float32)
    up = np.zeros((1, inter), np.float32)
    gate[0, ::32][:vals.size] = vals
    up[0, ::32][:vals.size] = 1.0
    h = synth.f32_to_bf16_bits(np.concatenate([gate, up], axis=1))
    q, s = fp.fp8_swiglu_quantize(to_dev_bf16(h), "mxfp8")
    torch.cuda.synchronize()
    assert_swiglu(q, s, to_f32(h), inter, "mxfp8", "swiglu isolated values")


def test_swiglu_far_negative_gates_each_alone():
    """Gates from -80 down to -110 with several up values, each alone in its
    1x128 group: y is a tiny normal or subnormal BF16 number (or -0), which
    the group's scale |y| / 448 exposes exactly."""
    g = np.arange(-80.0, -110.0, -0.125, dtype=np.float32)
    ups = np.array([1.0, -0.75, 100.0, 3.0e4], np.float32)
    vals = np.stack(np.meshgrid(g, ups, indexing="ij"), axis=-1).reshape(-1, 2)
    per_row = 16
    inter = 128 * per_row
    rows = -(-vals.shape[0] // per_row)
    gate = np.zeros((rows * per_row, 128), np.float32)
    up = np.zeros((rows * per_row, 128), np.float32)
    gate[:vals.shape[0], 0] = vals[:, 0]
    up[:vals.shape[0], 0] = vals[:, 1]
    h = synth.f32_to_bf16_bits(np.concatenate([gate.reshape(rows, inter), up.reshape(rows, inter)], axis=1))
    q, s = fp.fp8_swiglu_quantize(to_dev_bf16(h), "1x128")
    torch.cuda.synchronize()
    hf = to_f32(h)
    assert_swiglu(q, s, hf, inter, "1x128", "swiglu far-negative gates")
    # most of these are non-zero BF16 values (the float32 form would give -0)
    y = OM.swiglu_bf16(hf, inter)
    assert (y != 0).sum() > vals.shape[0] // 2


def test_swiglu_empty():
    h = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = fp.fp8_swiglu_quantize(h, "mxfp8")
    assert q.shape == (0, 128)


@pytest.mark.parametrize("gran", ("mxfp8", "1x128_pow2"))
def test_swiglu_full_moe_layer_sampled(gran):
    """The gate+up output of the MoE layer (131072 routed rows x 2 x 768):
    256 sampled rows against the oracle."""
    rows, inter = 131072, 768
    bits = synth.activations((rows, 2 * inter), seed=84)
    hd = to_dev_bf16(bits)
    q, s = fp.fp8_swiglu_quantize(hd, gran)
    torch.cuda.synchronize()
    pick = synth.rng(85).choice(rows, 256, replace=False)
    pick[:2] = [0, rows - 1]
    ti = torch.from_numpy(pick).cuda()
    assert_swiglu(q[ti], s[ti], to_f32(bits[pick]), inter, gran, f"swiglu full size {gran}")


# ---------------------------------------------------------------- the layer, step by step
def experts_deq(qw, sw):
    return [OG.dequant_mxfp8(np_u8(qw[e]), np_u8(sw[e])) for e in range(qw.shape[0])]


def test_moe_layer_chain():
    """gather+quantise -> grouped gate+up GEMM -> SwiGLU+quantise -> grouped
    down GEMM, MXFP8 throughout.  Each quantising step is compared bit for
    bit with the oracle fed the GPU's own input to that step; each GEMM with
    the oracle's exact product of the GPU's codes (tolerance of the GEMM
    contract)."""
    tokens, hidden, inter, experts, top_k = 512, 256, 128, 8, 2
    x = synth.activations((tokens, hidden), seed=91)
    w1 = synth.weights((experts, 2 * inter, hidden), seed=92)
    w2 = synth.weights((experts, hidden, inter), seed=93)
    idx, offsets = synth.moe_routing(tokens, experts, top_k, seed=94)
    off_d = torch.from_numpy(offsets).cuda()

    qa, sa = fp.fp8_quantize_gathered(to_dev_bf16(x), torch.from_numpy(idx).cuda(), "mxfp8")
    pq, ps = OM.quantize_gathered(to_f32(x), idx, "mxfp8")
    assert np.array_equal(np_u8(qa), pq) and np.array_equal(np_u8(sa), ps)

    qw1, sw1, _ = fp.fp8_quantize(to_dev_bf16(w1.reshape(-1, hidden)), "mxfp8")
    qw1 = qw1.view(experts, 2 * inter, hidden)
    sw1 = sw1.view(experts, 2 * inter, hidden // 32)
    h = fp.fp8_grouped_gemm(qa, sa, qw1, sw1, off_d, "mxfp8")
    torch.cuda.synchronize()
    ref_h = OG.grouped_gemm(OG.dequant_mxfp8(pq, ps), experts_deq(qw1, sw1), offsets)
    for e in range(experts):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            assert_gemm_close(bf16_to_f64(h)[lo:hi], ref_h[lo:hi])

    qy, sy = fp.fp8_swiglu_quantize(h, "mxfp8")
    h_bits = h.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_swiglu(qy, sy, to_f32(h_bits), inter, "mxfp8", "layer swiglu")
    # the down GEMM's reference takes the GPU's own codes (checked just above)
    pqy, psy = np_u8(qy), np_u8(sy)

    qw2, sw2, _ = fp.fp8_quantize(to_dev_bf16(w2.reshape(-1, inter)), "mxfp8")
    qw2 = qw2.view(experts, hidden, inter)
    sw2 = sw2.view(experts, hidden, inter // 32)
    out = fp.fp8_grouped_gemm(qy, sy, qw2, sw2, off_d, "mxfp8")
    torch.cuda.synchronize()
    ref_o = OG.grouped_gemm(OG.dequant_mxfp8(pqy, psy), experts_deq(qw2, sw2), offsets)
    for e in range(experts):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            assert_gemm_close(bf16_to_f64(out)[lo:hi], ref_o[lo:hi])
    assert fp.read_status() == 0
