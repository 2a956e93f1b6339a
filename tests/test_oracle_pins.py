"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks one oracle function against a closed form, a library
routine, an exhaustive table, a brute-force implementation or an invariant,
chosen so that a plausible slip (a dropped term, a wrong sign or index, a
transposed operand, a wrong tie-break) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_expert_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- codecs

def test_bf16_decode_exhaustive():
    L = oracle.lib()
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([L.orc_bf16_to_f64(int(b)) for b in bits[::7]])
    r = ref[::7]
    same = (got == r) | (np.isnan(got) & np.isnan(r))
    assert same.all()


def test_bf16_encode_matches_torch_rne():
    g = np.random.default_rng(1)
    u = g.integers(0, 1 << 32, size=1 << 18, dtype=np.uint64).astype(np.uint32)
    # plant exact midpoints (low half 0x8000) with odd and even kept halves
    u[:4096] = (u[:4096] & 0xFFFF0000) | 0x8000
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    got = oracle.bf16_encode(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_e4m3_decode_all_codes():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    same = (vals == ref) | (np.isnan(vals) & np.isnan(ref))
    assert same.all()
    # OCP E4M3 landmarks: largest finite, smallest normal, smallest subnormal
    assert vals[0x7E] == 448.0 and vals[0x08] == 2.0 ** -6 and vals[0x01] == 2.0 ** -9
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])


def test_e4m3_encode_rne_satfinite():
    finite = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    grid = np.unique(finite[np.isfinite(finite) & (finite >= 0)])
    mids = (grid[:-1] + grid[1:]) / 2                       # exact ties
    g = np.random.default_rng(2)
    rnd = np.concatenate([g.normal(0, s, 20000) for s in (1e-3, 0.1, 3, 60, 400)])
    x = np.concatenate([grid, mids, -mids, rnd, [448.0, 449.0, 470.0, 1e6, -1e6, 0.0]]).astype(np.float32)
    got = oracle.e4m3_encode(x)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # ties go to the even code
    codes_mid = oracle.e4m3_encode(mids.astype(np.float32))
    assert (codes_mid % 2 == 0).all()
    # saturation instead of NaN
    assert oracle.e4m3_encode(np.array([1e9, -1e9], np.float32)).tolist() == [0x7E, 0xFE]


def test_quant_blocks_definition():
    g = np.random.default_rng(3)
    w = g.normal(0, 1, (256, 384)).astype(np.float32)
    w[:128, 128:256] *= 1e-3                     # blocks with very different scales
    w[128:, :128] = 0.0                          # an all-zero block -> scale 1, codes 0
    q, s = oracle.quant_blocks(w, 128, 128)
    assert s.shape == (2, 3)
    for bi in range(2):
        for bj in range(3):
            blk = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            if amax == 0:
                assert s[bi, bj] == 1.0
                assert (q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128] == 0).all()
                continue
            assert s[bi, bj] == np.float32(amax / np.float32(448.0))
            inv = np.float32(np.float32(448.0) / amax)
            ref = torch.from_numpy((blk * inv).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128], ref)
            # the block's largest magnitude maps to the largest code
            assert np.abs(oracle.e4m3_decode(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128])).max() == 448.0
    # dequantised values stay within half a code step (relative 2^-4) of w
    deq = oracle.e4m3_decode(q) * np.repeat(np.repeat(s, 128, 0), 128, 1)
    nz = np.abs(w) > 1e-2 * np.repeat(np.repeat(s * 448, 128, 0), 128, 1)
    assert np.all(np.abs(deq - w)[nz] <= np.abs(w)[nz] * 2.0 ** -4 + 1e-12)


def _torch_quant_row_128(v, width=128):
    """Independent per-row, per-128-column E4M3 quantiser (torch's cast),
    returned as code value * scale: s = amax/448, code = e4m3(fp32(v * fp32(448/amax))),
    an all-zero group keeps scale 1.  (`width` only serves to build the
    wrong variants the pin must tell apart.)"""
    v = np.asarray(v, np.float32)
    rows, cols = v.shape
    out = np.empty((rows, cols), np.float64)
    for c0 in range(0, cols, width):
        grp = v[:, c0:c0 + width]
        amax = np.abs(grp).max(axis=1).astype(np.float32)
        zero = amax == 0
        a = np.where(zero, np.float32(1), amax).astype(np.float32)
        scale = np.where(zero, np.float32(1), (a / np.float32(448)).astype(np.float32)).astype(np.float32)
        inv = np.where(zero, np.float32(1), (np.float32(448) / a).astype(np.float32)).astype(np.float32)
        p = (grp * inv[:, None]).astype(np.float32)
        codes = torch.from_numpy(p).to(torch.float8_e4m3fn).double().numpy()
        out[:, c0:c0 + width] = codes * scale.astype(np.float64)[:, None]
    return out


def test_quant_row_128_definition():
    """The FP8 layer's activation quantiser (x before the gate/up GEMM, h
    before the down GEMM): one scale per row and 128 columns.  Groups whose
    amax spans four decades, an all-zero group and exact E4M3 ties make a
    group width of 256, a whole-row amax or a wrong tie rule fail."""
    g = np.random.default_rng(21)
    rows, cols = 6, 768
    v = g.normal(0, 1, (rows, cols)).astype(np.float32)
    decades = np.array([1e-3, 1e-1, 1e1, 1e-2, 1.0, 1e2], np.float32)
    for r in range(rows):
        v[r] *= np.repeat(np.roll(decades, r), 128)
    v[2, 256:384] = 0.0                                   # an all-zero group
    # a group with amax exactly 448 (scale 1): E4M3 midpoints tie to even
    grid = oracle.e4m3_decode(np.arange(0x38, 0x50, dtype=np.uint8))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    v[4, 128:128 + len(mids)] = mids
    v[4, 128 + len(mids):256] = 0.25
    v[4, 255] = 448.0
    got = oracle.quant_rows_128(v)
    ref = _torch_quant_row_128(v)
    assert np.array_equal(got, ref)
    assert (got[2, 256:384] == 0).all()
    codes_mid = oracle.e4m3_encode(mids)
    assert np.array_equal(got[4, 128:128 + len(mids)], oracle.e4m3_decode(codes_mid))
    assert (codes_mid % 2 == 0).all()
    # the plausible slips give different values on these rows
    for width in (256, cols):                    # 256-wide groups; one amax per row
        assert (_torch_quant_row_128(v, width) != got).mean() > 0.25


def test_fp8_single_expert_layer_quantises_x_and_h_per_128_group():
    """E = 1, k = 1 FP8 layer: x is quantised per token per 128 columns
    before the gate/up projections and h (rounded to fp32) before the down
    projection, weights are the 128x128 block codes times their scales.
    Checked against numpy matmuls over torch's E4M3 cast."""
    shape = synth.LayerShape("t", 5, 256, 1, 256, 1, "fp8")
    inp = synth.make_inputs(shape, seed=22)
    exq = oracle.Experts.quantised(inp["w_gate"], inp["w_up"], inp["w_down"])
    x = inp["x"]
    out, y = oracle.moe_tokens(x, np.zeros((5, 1), np.int32), np.ones((5, 1)), exq, want_y=True)

    def deq(q, s):
        return oracle.e4m3_decode(q) * np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)

    xd = _torch_quant_row_128(x.float().numpy())
    ref = np.zeros((5, 256))
    for grp in range(2):
        a = xd @ deq(exq.wg[grp], exq.sg[grp]).T
        u = xd @ deq(exq.wu[grp], exq.su[grp]).T
        h = (a / (1 + np.exp(-a)) * u).astype(np.float32)
        yg = _torch_quant_row_128(h) @ deq(exq.wd[grp], exq.sd[grp]).T
        assert np.allclose(y[:, 0 if grp == 0 else 1], yg, rtol=1e-12, atol=1e-12)
        ref += yg
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- routing

def _brute_topk(z, k):
    """Independent top-k: a full stable sort by (-z, expert index)."""
    T, E = z.shape
    idx = np.empty((T, k), np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-z[t, e], e))
        idx[t] = order[:k]
    return idx


@pytest.mark.parametrize("T,E,k", [(50, 16, 2), (40, 32, 10), (20, 8, 8), (10, 5, 1)])
def test_topk_vs_brute_force_with_ties(T, E, k):
    z = synth.tie_logits(T, E, seed=T + E).double().numpy()
    idx, w = oracle.topk(z, k)
    assert np.array_equal(idx, _brute_topk(z, k))
    assert np.allclose(w.sum(1), 1.0, atol=1e-15, rtol=0)
    assert (np.diff(w, axis=1) <= 1e-18).all()     # slot order: descending weight


def test_topk_weights_closed_forms():
    g = np.random.default_rng(4)
    z = g.normal(0, 2, (30, 12))
    _, w1 = oracle.topk(z, 1)
    assert (w1 == 1.0).all()
    idx, wE = oracle.topk(z, 12)
    from scipy.special import softmax
    full = softmax(z, axis=1)
    assert np.allclose(np.take_along_axis(full, idx, 1), wE, rtol=1e-14, atol=0)
    # renormalising the full softmax over the chosen set gives the same weights
    idx3, w3 = oracle.topk(z, 3)
    sel = np.take_along_axis(full, idx3, 1)
    assert np.allclose(sel / sel.sum(1, keepdims=True), w3, rtol=1e-13, atol=0)


def test_blob_round_trip():
    g = np.random.default_rng(5)
    z = g.normal(size=(1024, 64))
    idx, w = oracle.topk(z, 10)
    blob = oracle.pack_blob(idx, w)
    assert blob.shape == (2, 1024, 10) and blob.dtype == np.int32
    assert np.array_equal(blob[0], idx)
    assert np.array_equal(blob[1].view(np.float32), w.astype(np.float32))


def test_compact_word_matches_independent_packing():
    """One-word blob: low 16 bits the index, high 16 bits bf16(w); checked
    against numpy bit twiddling over torch's bf16 rounding."""
    g = np.random.default_rng(8)
    idx, w = oracle.topk(g.normal(size=(500, 512)), 10)
    words = oracle.pack_words(idx, w).view(np.uint32)
    wb = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = (idx.astype(np.uint32) & 0xFFFF) | (wb.astype(np.uint32) << 16)
    assert np.array_equal(words, ref)
    assert np.array_equal((words & 0xFFFF).astype(np.int32), idx)
    back = (words >> 16).astype(np.uint32) << 16
    assert np.allclose(back.view(np.float32), w, rtol=2.0 ** -8, atol=0)


# ------------------------------------------------------------ permutation

@pytest.mark.parametrize("T,E,k,seed", [(64, 16, 2, 0), (300, 32, 4, 1), (7, 5, 5, 2), (1, 3, 1, 3)])
def test_permute_invariants_and_stable_sort(T, E, k, seed):
    g = np.random.default_rng(seed)
    z = g.normal(size=(T, E)) + np.log(np.arange(1, E + 1))[g.permutation(E)]
    idx, _ = oracle.topk(z, k)
    counts, offsets, inv, src = oracle.permute(idx, E)
    assert counts[:E].sum() == T * k and counts[E] == T
    assert offsets[0] == 0 and offsets[E] == T * k and offsets[E + 1] == T * k + T
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(inv), np.arange(T * k))          # bijection
    assert np.array_equal(src[inv], np.repeat(np.arange(T), k))
    assert np.array_equal(src[T * k:], np.arange(T))
    # independent: a stable argsort of the flat expert ids gives the positions
    order = np.argsort(idx.reshape(-1), kind="stable")
    rank = np.empty(T * k, np.int64)
    rank[order] = np.arange(T * k)
    assert np.array_equal(inv, rank)
    # every position lies inside its expert's segment
    e_of = idx.reshape(-1)
    assert ((inv >= offsets[e_of]) & (inv < offsets[e_of + 1])).all()


def test_identity_experts_permute_unpermute():
    """y_e = x for every expert, shared expert off: the combine returns x."""
    g = np.random.default_rng(6)
    T, E, k, D = 97, 12, 3, 24
    x = g.normal(size=(T, D))
    idx, w = oracle.topk(g.normal(size=(T, E)), k)
    counts, offsets, inv, src = oracle.permute(idx, E)
    y = np.zeros((T * k + T, D))
    y[:T * k] = x[src[:T * k]]
    out = oracle.unpermute(y, w, inv, T, k)
    assert np.allclose(out, x, rtol=0, atol=1e-14)
    # shared expert alone (routed outputs zero) gives the shared rows back
    y2 = np.zeros_like(y)
    y2[T * k:] = x
    assert np.array_equal(oracle.unpermute(y2, w, inv, T, k), x)


# ------------------------------------------------------------ expert FFN

def _np_swiglu(x, wg, wu, wd):
    a = x @ wg.T
    u = x @ wu.T
    return (a / (1 + np.exp(-a)) * u) @ wd.T


def test_single_expert_is_dense_swiglu():
    """E = 1, k = 1: out = shared(x) + expert0(x), each a dense SwiGLU FFN."""
    shape = synth.LayerShape("t", 9, 64, 1, 32, 1, "f32")
    inp = synth.make_inputs(shape, seed=11)
    ex = oracle.Experts("f32", inp["w_gate"], inp["w_up"], inp["w_down"])
    out, idx, w = oracle.moe_layer(inp["x"], inp["w_router"], None, ex, 1)
    assert (idx == 0).all() and (w == 1.0).all()
    x = inp["x"].double().numpy()
    wg, wu, wd = (inp[n].double().numpy() for n in ("w_gate", "w_up", "w_down"))
    ref = _np_swiglu(x, wg[0], wu[0], wd[0]) + _np_swiglu(x, wg[1], wu[1], wd[1])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_topk_equal_E_is_dense_softmax_mixture(dtype):
    shape = synth.LayerShape("t", 11, 64, 6, 32, 6, dtype, 1.0)
    inp = synth.make_inputs(shape, seed=12)
    ex = oracle.Experts(dtype, inp["w_gate"], inp["w_up"], inp["w_down"])
    out, _, _ = oracle.moe_layer(inp["x"], inp["w_router"], inp["b_router"], ex, 6)
    x = inp["x"].double().numpy()
    z = x @ inp["w_router"].double().numpy().T + inp["b_router"].double().numpy()
    from scipy.special import softmax
    p = softmax(z, axis=1)
    wg, wu, wd = (inp[n].double().numpy() for n in ("w_gate", "w_up", "w_down"))
    ref = _np_swiglu(x, wg[6], wu[6], wd[6])
    for e in range(6):
        ref += p[:, e:e + 1] * _np_swiglu(x, wg[e], wu[e], wd[e])
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sparse_layer_is_the_dense_mixture_when_the_rest_carry_no_mass(dtype):
    """k < E: a random set S of k experts gets router bias 0 and every other
    expert -1000, so the full softmax gives the others exactly zero mass in
    fp64 (exp(-1000) underflows).  The sparse layer -- choose the top k,
    softmax over the chosen, combine -- must then equal the dense softmax
    mixture over all E experts plus the shared expert, computed with numpy and
    scipy.  A wrong expert chosen, a weight paired with another slot's expert
    or a missing renormalisation all move the result."""
    E, k = 12, 4
    shape = synth.LayerShape("t", 10, 64, E, 32, k, dtype, 1.0)
    inp = synth.make_inputs(shape, seed=21)
    chosen = np.random.default_rng(5).permutation(E)[:k]
    bias = np.full(E, -1000.0, dtype=np.float32)
    bias[chosen] = 0.0
    b = torch.from_numpy(bias)
    ex = oracle.Experts(dtype, inp["w_gate"], inp["w_up"], inp["w_down"])
    out, idx, _ = oracle.moe_layer(inp["x"], inp["w_router"], b, ex, k)
    assert all(set(row) == set(chosen.tolist()) for row in np.asarray(idx).tolist())
    x = inp["x"].double().numpy()
    z = x @ inp["w_router"].double().numpy().T + bias.astype(np.float64)
    from scipy.special import softmax
    p = softmax(z, axis=1)
    wg, wu, wd = (inp[n].double().numpy() for n in ("w_gate", "w_up", "w_down"))
    ref = _np_swiglu(x, wg[E], wu[E], wd[E])
    for e in range(E):
        ref += p[:, e:e + 1] * _np_swiglu(x, wg[e], wu[e], wd[e])
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_layer_equivariances():
    shape = synth.SMALL_F32.with_tokens(23)
    inp = synth.make_inputs(shape, seed=13)
    ex = oracle.Experts("f32", inp["w_gate"], inp["w_up"], inp["w_down"])
    out, idx, w = oracle.moe_layer(inp["x"], inp["w_router"], None, ex, shape.top_k)
    # token order: permuting tokens permutes rows, bit for bit
    perm = np.random.default_rng(0).permutation(23)
    out_p, _, _ = oracle.moe_layer(inp["x"][perm], inp["w_router"], None, ex, shape.top_k)
    assert np.array_equal(out_p, out[perm])
    # expert relabelling: permute router rows and expert groups together
    E = shape.E
    rl = np.random.default_rng(1).permutation(E)
    gperm = np.concatenate([rl, [E]])
    ex2 = oracle.Experts("f32", inp["w_gate"][gperm], inp["w_up"][gperm], inp["w_down"][gperm])
    out_r, idx_r, _ = oracle.moe_layer(inp["x"], inp["w_router"][rl], None, ex2, shape.top_k)
    assert np.array_equal(rl[idx_r], idx)
    assert np.array_equal(out_r, out)
    # y slots: the combine of the per-expert outputs is the layer output
    out_t, y = oracle.moe_tokens(inp["x"], idx, w, ex, want_y=True)
    assert np.array_equal(out_t, out)
    comb = y[:, shape.top_k] + sum(w[:, j:j + 1] * y[:, j] for j in range(shape.top_k))
    assert np.allclose(comb, out, rtol=1e-14, atol=1e-14)


def test_fp8_mode_tracks_unquantised_layer():
    """FP8 mode stays within E4M3 error of the fp64 layer on the unquantised
    weights, and is not identical to it (quantisation happened).  E4M3 keeps 3
    mantissa bits (relative step 2^-3), so x, w, h and w_down each carry a few
    per cent of rounding: the rms error of the layer lands near 6 % of the
    output rms.  Block scales spread over four decades, so a transposed or
    misplaced scale index lands far outside the bound."""
    shape = synth.LayerShape("t", 13, 256, 4, 256, 2, "fp8", 1.0)
    inp = synth.make_inputs(shape, seed=14)
    g = torch.Generator().manual_seed(5)
    def spread(w):
        G, R, C = w.shape
        f = 10.0 ** torch.randint(-2, 2, (G, R // 128, C // 128), generator=g).float()
        return w * f.repeat_interleave(128, 1).repeat_interleave(128, 2)
    wg, wu, wd = spread(inp["w_gate"]), spread(inp["w_up"]), spread(inp["w_down"])
    exq = oracle.Experts.quantised(wg, wu, wd)
    out8, idx, w = oracle.moe_layer(inp["x"], inp["w_router"], inp["b_router"], exq, 2)
    ex32 = oracle.Experts("f32", wg, wu, wd)
    x32 = inp["x"].float()
    ref = oracle.moe_tokens(x32, idx, w, ex32)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.sqrt(np.mean((out8 - ref) ** 2))
    assert 1e-3 * rms < err <= 0.12 * rms
    # a misplaced scale (transposed block grid of the gate weights) breaks it
    bad = oracle.Experts("fp8", exq.wg, exq.wu, exq.wd, np.ascontiguousarray(exq.sg.transpose(0, 2, 1)), exq.su, exq.sd)
    out_bad = oracle.moe_tokens(inp["x"], idx, w, bad)
    assert np.sqrt(np.mean((out_bad - ref) ** 2)) > 0.5 * rms
    bad = oracle.Experts("fp8", exq.wg, exq.wu, exq.wd, exq.sg, exq.su, np.ascontiguousarray(exq.sd[::-1]))
    out_bad = oracle.moe_tokens(inp["x"], idx, w, bad)
    assert np.sqrt(np.mean((out_bad - ref) ** 2)) > 0.5 * rms


def test_fp8_exact_grid_inputs_are_lossless():
    """Inputs already on the E4M3 grid with every 128-group holding +-448
    quantise with scale 1 and no rounding: FP8-mode routed outputs then equal
    the fp32-mode ones up to the h quantisation, which the shared expert with
    an all-zero down projection isolates (its output must be exactly 0)."""
    D, I = 128, 128
    grid = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    g = np.random.default_rng(7)
    x = g.choice(grid, (3, D)) * g.choice([-1, 1], (3, D))
    x[:, 0] = 448.0
    xq = oracle.as_bits(torch.from_numpy(x).to(torch.bfloat16))[0]
    assert np.array_equal(torch.from_numpy(xq.view(np.int16)).view(torch.bfloat16).double().numpy(), x)
    wg = g.choice(grid, (2, I, D)) * 2.0 ** -9
    wg[:, 0, 0] = 448.0
    wu = wg.copy()
    wd = np.zeros((2, D, I)); wd[0] = g.choice(grid, (D, I)); wd[0, 0, 0] = 448.0
    exq = oracle.Experts.quantised(wg.astype(np.float32), wu.astype(np.float32), wd.astype(np.float32))
    assert (exq.sg == 1.0).all() and (exq.su == 1.0).all() and exq.sd[0, 0, 0] == 1.0
    out = oracle.moe_tokens(torch.from_numpy(x).to(torch.bfloat16), np.zeros((3, 1), np.int32),
                            np.ones((3, 1)), exq, want_y=True)[1]
    assert (out[:, 1] == 0).all()                               # shared: zero down weights


# ---------------------------------------------------------- page constants

def test_workloads_use_page_constants():
    c = json.load(open(os.path.join(GOLDEN, "layer_constants.json")))
    for s in (synth.DECODE_BF16, synth.BATCHED_DECODE_BF16, synth.PREFILL_BF16, synth.PREFILL_FP8):
        assert (s.D, s.E, s.I, s.top_k) == (c["hidden_D"]["value"], c["routed_experts_E"]["value"],
                                            c["expert_intermediate_I"]["value"], c["top_k"]["value"])
    assert synth.BATCHED_DECODE_BF16.T == c["blob_plane_shape"]["value"][0]
    assert c["blob_planes"]["value"] == 2 and c["blob_word_bits"]["value"] == 32


def test_tiny_workload_runs_in_oracle():
    shape = synth.TINY_F32
    inp = synth.make_inputs(shape, seed=0)
    ex = oracle.Experts("f32", inp["w_gate"], inp["w_up"], inp["w_down"])
    out, idx, w = oracle.moe_layer(inp["x"], inp["w_router"], None, ex, shape.top_k)
    assert out.shape == (64, 256) and np.isfinite(out).all()
    counts, *_ = oracle.permute(idx, shape.E)
    assert counts[:shape.E].sum() == 64 * 2
