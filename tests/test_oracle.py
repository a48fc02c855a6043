"""Pins for the CPU oracle: every check here comes from somewhere other than
the oracle itself -- a hand-derived fixture under tests/golden/, a library
routine (numpy matmul / stable argsort, scipy softmax, torch dtype casts),
brute-force enumeration on tiny inputs, a closed form, or an invariant the
pages state.  CPU only.
"""
import itertools
import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

import moe_inputs as mi
import oracle
from conftest import golden_dict, read_golden


def widen(bits):
    return oracle.bf16_bits_to_f64_array(bits)


def ref_logits(X, W, bias=None):
    """Library matmul of the exactly widened bf16 operands (fp64)."""
    L = widen(mi.bf16_bits(X)) @ widen(mi.bf16_bits(W))
    if bias is not None:
        L = L + bias.numpy().astype(np.float64)[None, :]
    return L


def to_bits(values):
    return mi.bf16_bits(torch.tensor(values, dtype=torch.float32).to(torch.bfloat16))


# ---------------------------------------------------------------- formats

def test_bf16_widening_matches_torch():
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    mine = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(t)
    assert np.array_equal(mine[finite], t[finite])
    assert np.array_equal(np.isnan(mine), np.isnan(t))


def test_bf16_rounding_matches_torch_on_fp32_values():
    # fp32 values are exact in fp64, so torch's float32 -> bf16 RNE is a direct check
    rng = np.random.default_rng(0)
    raw = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = raw.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([oracle.f64_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_rounding_is_single_rounding_from_fp64():
    # 1 + 2^-8 is the tie between 1 and 1 + 2^-7; anything above it rounds up.
    assert oracle.f64_to_bf16(1.0 + 2.0**-8) == 0x3F80           # tie -> even (1.0)
    assert oracle.f64_to_bf16(1.0 + 2.0**-8 + 2.0**-40) == 0x3F81  # just above -> up
    assert oracle.f64_to_bf16(1.0 + 3 * 2.0**-8) == 0x3F82       # tie -> even (m=2)
    assert oracle.f64_to_bf16(2.0**-133) == 0x0001               # smallest subnormal
    assert oracle.f64_to_bf16(2.0**-134) == 0x0000               # tie with zero -> even
    # max bf16 = 255 * 2^120; the overflow threshold is 255.5 * 2^120 = 3.396177...e38
    assert oracle.f64_to_bf16(3.3961e38) == 0x7F7F               # below threshold -> max
    assert oracle.f64_to_bf16(3.3962e38) == 0x7F80               # past max + half ulp -> inf


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    assert np.array_equal(np.isnan(mine), np.isnan(t))
    ok = ~np.isnan(t)
    assert np.array_equal(mine[ok], t[ok])
    assert np.nanmax(mine) == 448.0 and np.nanmin(mine) == -448.0


def test_e4m3_roundtrip_all_finite_codes():
    for c in range(256):
        v = oracle.e4m3_to_f64(c)
        if math.isnan(v):
            continue
        assert oracle.f64_to_e4m3(v) == c, (c, v)


def test_e4m3_golden_points():
    for value, code in read_golden("e4m3_points.txt"):
        assert oracle.f64_to_e4m3(float(value)) == int(code, 16), value
    assert oracle.f64_to_e4m3(float("nan")) == 0x7F


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-448, 448, 5000), rng.normal(0, 1, 5000),
                           rng.normal(0, 0.01, 5000)]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.f64_to_e4m3(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(mine, ref)


def test_fp8_block_scale_golden():
    for amax, s in read_golden("fp8_block_scale.txt"):
        assert oracle.fp8_block_scale(float(amax)) == float(s), amax


def test_fp8_block_scale_is_smallest_pow2_not_below_t():
    # closed form: s = 2^ceil(log2 t) with t the fp32 product of the page's rule
    rng = np.random.default_rng(2)
    for amax in np.concatenate([rng.uniform(0, 10, 500), 10.0 ** rng.uniform(-6, 30, 500)]):
        s = oracle.fp8_block_scale(float(amax))
        m, e = math.frexp(s)
        assert m == 0.5, s                    # a power of two
        a = max(np.float32(amax), np.float32(1e-4))
        t = float(np.float32(a) * np.float32(1.0 / 448.0))
        assert s >= t and s / 2 < t, (amax, s, t)


def test_ue8m0_block_scale_golden():
    for amax, b in read_golden("ue8m0_block_scale.txt"):
        assert oracle.ue8m0_block_scale(float(amax)) == int(b), amax


def test_ue8m0_block_scale_rounds_up_and_matches_fp32_branch():
    # closed form of round-toward-+inf to a power of two: 2^(b-127) >= t > 2^(b-128);
    # and the two branches of the page's rule give the same scale value
    rng = np.random.default_rng(3)
    for amax in np.concatenate([rng.uniform(0, 10, 500), 10.0 ** rng.uniform(-6, 30, 500)]):
        b = oracle.ue8m0_block_scale(float(amax))
        a = max(np.float32(amax), np.float32(1e-4))
        t = float(np.float32(a) * np.float32(1.0 / 448.0))
        assert 2.0 ** (b - 127) >= t and 2.0 ** (b - 128) < t, (amax, b, t)
        assert 2.0 ** (b - 127) == oracle.fp8_block_scale(float(amax))


def test_permute_ue8m0_matches_fp32_scale_path():
    N, H, E, K = 30, 384, 8, 3
    X = mi.random_bf16((N, H), seed=31, scale=3.0)
    X[0, :128] = 0.0
    X[1, 128:256] *= 1e-6
    X[2, 256:] *= 500.0
    idx = mi.random_topk_idx(N, E, K, seed=32).numpy()
    _, _, row_map, _ = oracle.dispatch(idx, E)
    _, Xq, Xs = oracle.permute(mi.bf16_bits(X), row_map, K, fp8=True)
    Xq8, Xs8 = oracle.permute_ue8m0(mi.bf16_bits(X), row_map, K)
    assert Xs8.dtype == np.uint8
    assert np.array_equal(Xq8, Xq)
    assert np.array_equal(np.ldexp(1.0, Xs8.astype(np.int32) - 127), Xs.astype(np.float64))


# ---------------------------------------------------------------- expert-parallel dispatch metadata

def brute_force_ep(idx, E, R):
    """Plain-Python statement of the dedup'd send layout: rows are the sorted set of (rank, token)."""
    N, K = idx.shape
    P = E // R
    pairs = sorted({(int(e) // P, n) for n in range(N) for e in idx[n]})
    row = {pr: i for i, pr in enumerate(pairs)}
    rank_counts = [sum(1 for r, _ in pairs if r == q) for q in range(R)]
    rank_offsets = [0] + list(itertools.accumulate(rank_counts))
    send_token = [n for _, n in pairs]
    slot_send_row = [row[(int(idx[n, k]) // P, n)] for n in range(N) for k in range(K)]
    return rank_counts, rank_offsets, send_token, slot_send_row


@pytest.mark.parametrize("N,E,K,R", [(1, 4, 1, 2), (9, 8, 3, 4), (20, 16, 4, 4), (33, 12, 5, 3), (50, 64, 8, 8),
                                     (17, 6, 2, 6), (25, 10, 4, 1)])
def test_dispatch_ep_matches_brute_force(N, E, K, R):
    idx = mi.random_topk_idx(N, E, K, seed=N * E + R).numpy()
    o = oracle.dispatch_ep(idx, E, R)
    rc, ro, st, ssr = brute_force_ep(idx, E, R)
    assert o["rank_counts"].tolist() == rc and o["rank_offsets"].tolist() == ro
    assert o["send_token"].tolist() == st and o["slot_send_row"].tolist() == ssr
    P = E // R
    counts = np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(o["send_meta"][:, 0], rc)
    assert np.array_equal(o["send_meta"][:, 1:].ravel(), counts)
    # expanding a rank's received rows by expand_idx gives, row by row, the token of every
    # expert-ordered slot of that rank
    for q in range(N * K):
        s = o["src_slot"][q]
        r = idx.ravel()[s] // P
        assert 0 <= o["expand_idx"][q] < rc[r]
        assert st[ro[r] + o["expand_idx"][q]] == s // K


def test_dispatch_ep_special_cases():
    N, E, K = 40, 16, 4
    idx = mi.random_topk_idx(N, E, K, seed=5).numpy()
    # one rank: every token once, in order; each slot's row is its token
    o = oracle.dispatch_ep(idx, E, 1)
    assert o["rank_counts"].tolist() == [N] and o["send_token"].tolist() == list(range(N))
    assert np.array_equal(o["slot_send_row"], np.arange(N * K) // K)
    assert np.array_equal(o["expand_idx"], o["src_slot"] // K)
    # one expert per rank: nothing to deduplicate (the K experts of a token are distinct),
    # so the rank order is the expert order
    o = oracle.dispatch_ep(idx, E, E)
    assert np.array_equal(o["slot_send_row"], o["row_map"])
    assert np.array_equal(o["rank_counts"], o["counts"])
    assert np.array_equal(o["expand_idx"], np.arange(N * K) - np.repeat(o["offsets"][:-1], o["counts"]))


# ---------------------------------------------------------------- router statistics

def test_logsumexp_matches_scipy_and_special_cases():
    from scipy.special import logsumexp as sp_lse
    X, W, bias = mi.make_route_inputs(64, 128, 32, seed=11, skew=True)
    _, _, L = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), bias.numpy(), 2, want_logits=True)
    lse = oracle.logsumexp(L)
    assert np.allclose(lse, sp_lse(L, axis=1), rtol=0, atol=1e-12)
    # equal logits: c + log(E); one expert: the logit itself; NaN counts as -inf; all -inf gives -inf
    E = 16
    Lc = np.full((3, E), 2.5)
    Lc[1, :] = -7.0
    Lc[2, 3] = np.nan
    Lc[2, 4:] = -np.inf
    got = oracle.logsumexp(Lc)
    assert got[0] == pytest.approx(2.5 + math.log(E), abs=1e-15)
    assert got[1] == pytest.approx(-7.0 + math.log(E), abs=1e-15)
    assert got[2] == pytest.approx(2.5 + math.log(3), abs=1e-15)
    assert oracle.logsumexp(np.array([[1.25]]))[0] == 1.25
    assert oracle.logsumexp(np.full((1, 4), -np.inf))[0] == -np.inf


def test_load_stats_hand_example():
    # counts 1,2,3,4: mean 2.5, max/mean 1.6; p95 at position 2.85 -> 3 + 0.85 = 3.85 -> 1.54
    st = oracle.load_stats(np.array([3, 1, 4, 2], np.int32), np.array([1.0, -2.0, 3.0]), 1e-3)
    assert st[0] == pytest.approx(1.6, abs=1e-15)
    assert st[1] == pytest.approx(3.85 / 2.5, abs=1e-15)
    assert st[2] == pytest.approx(1e-3 * (1 + 4 + 9) / 3, abs=1e-18)
    assert st[3] == 2.5
    # no lse: no z-loss; all counts zero: ratios 0; a uniform load: ratios 1
    assert oracle.load_stats(np.zeros(8, np.int32))[0:3].tolist() == [0.0, 0.0, 0.0]
    assert oracle.load_stats(np.full(8, 5, np.int32))[0:2].tolist() == [1.0, 1.0]


def test_load_stats_matches_numpy_percentile():
    rng = np.random.default_rng(12)
    for E in (1, 2, 7, 64, 256):
        c = rng.integers(0, 1000, E).astype(np.int32)
        lse = rng.normal(size=50)
        st = oracle.load_stats(c, lse, 1e-3)
        mean = c.sum() / E
        assert st[0] == pytest.approx(c.max() / mean, rel=1e-14)
        assert st[1] == pytest.approx(np.percentile(c, 95) / mean, rel=1e-14)
        assert st[2] == pytest.approx(1e-3 * np.mean(lse ** 2), rel=1e-14)


# ---------------------------------------------------------------- route

def test_route_golden_ties():
    g = golden_dict("route_ties.txt")
    N, H, E, K = (int(g[k][0]) for k in ("N", "H", "E", "K"))
    X = to_bits([float(v) for v in g["X"]]).reshape(N, H)
    W = to_bits([float(v) for v in g["W"]]).reshape(H, E)
    idx, w, L = oracle.route(X, W, None, K, renorm=True, want_logits=True)
    assert np.array_equal(L.ravel(), np.array(g["logits"], dtype=np.float64))
    assert np.array_equal(idx.ravel(), np.array(g["topk_idx"], dtype=np.int32))
    assert np.allclose(w.ravel(), np.array(g["topk_w_renorm"], dtype=np.float64), atol=2e-7)
    _, w2 = oracle.route(X, W, None, K, renorm=False)
    assert np.allclose(w2.ravel(), np.array(g["topk_w_plain"], dtype=np.float64), atol=2e-7)


@pytest.mark.parametrize("seed", range(3))
def test_route_logits_match_library_matmul(seed):
    X, W, _ = mi.make_route_inputs(37, 96, 24, seed)
    bias = torch.linspace(-1, 1, 24)
    _, _, L = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), bias.numpy(), 3, want_logits=True)
    ref = ref_logits(X, W, bias)
    assert np.max(np.abs(L - ref)) < 1e-12


@pytest.mark.parametrize("E,K", [(5, 1), (6, 2), (7, 3), (8, 4), (10, 4), (9, 2)])
def test_route_topk_brute_force(E, K):
    X, W, _ = mi.make_route_inputs(40, 32, E, seed=E * 10 + K)
    idx, w = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, K)
    L = ref_logits(X, W)
    for n in range(L.shape[0]):
        best = max(itertools.combinations(range(E), K), key=lambda c: sum(L[n, list(c)]))
        assert set(idx[n]) == set(best)
        assert all(L[n, idx[n, k]] >= L[n, idx[n, k + 1]] for k in range(K - 1))


def test_route_integer_ties_lower_index_wins():
    # integer-valued bf16 operands give exact integer logits with many ties
    g = torch.Generator().manual_seed(5)
    X = torch.randint(-2, 3, (64, 8), generator=g).to(torch.bfloat16)
    W = torch.randint(-1, 2, (8, 12), generator=g).to(torch.bfloat16)
    for K in (1, 3, 6, 12):
        idx, _ = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, K)
        L = ref_logits(X, W)
        E = L.shape[1]
        for n in range(L.shape[0]):
            order = np.lexsort((np.arange(E), -L[n]))  # by -L, then by index
            assert np.array_equal(idx[n], order[:K])


def test_route_k1_is_argmax_and_kE_is_full_descending_sort():
    X, W, _ = mi.make_route_inputs(50, 64, 16, seed=3)
    L = ref_logits(X, W)
    idx1, w1 = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, 1)
    assert np.array_equal(idx1[:, 0], np.argmax(L, axis=1))
    assert np.all(w1 == 1.0)
    idxE, _ = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, 16)
    assert np.array_equal(idxE, np.argsort(-L, axis=1, kind="stable"))


@pytest.mark.parametrize("renorm", [True, False])
def test_route_weights_closed_form(renorm):
    X, W, _ = mi.make_route_inputs(64, 128, 32, seed=4)
    bias = mi.zipf_bias(32)
    idx, w, P = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), bias.numpy(), 4,
                             renorm=renorm, want_probs=True)
    L = ref_logits(X, W, bias)
    assert np.allclose(P, softmax(L, axis=1), atol=1e-14, rtol=1e-12)
    sel = np.take_along_axis(L, idx.astype(np.int64), axis=1)
    if renorm:
        ref = softmax(sel, axis=1)          # renorm == softmax over the selected logits
        assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    else:
        ref = np.take_along_axis(softmax(L, axis=1), idx.astype(np.int64), axis=1)
    assert np.max(np.abs(w - ref)) < 1e-7
    assert np.all(np.diff(w, axis=1) <= 0)  # non-increasing in k


def test_route_bias_shifts_selection():
    X, W, _ = mi.make_route_inputs(128, 64, 16, seed=6)
    huge = np.zeros(16, np.float32)
    huge[7] = 1e3
    idx, w = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), huge, 2)
    assert np.all(idx[:, 0] == 7)
    assert np.all(w[:, 0] > 0.999)


def test_route_nan_logit_counts_as_minus_inf():
    X, W, _ = mi.make_route_inputs(16, 32, 8, seed=7)
    bias = np.zeros(8, np.float32)
    bias[0] = np.nan
    idx, _ = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), bias, 8)
    assert np.all(idx[:, -1] == 0)          # the NaN expert is taken last
    idx2, _ = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), bias, 3)
    assert not np.any(idx2 == 0)


def test_route_rejects_bad_k():
    X, W, _ = mi.make_route_inputs(4, 8, 4, seed=0)
    with pytest.raises(oracle.OracleError):
        oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, 5)


# ---------------------------------------------------------------- dispatch

def brute_force_dispatch(idx, E):
    N, K = idx.shape
    row_map = np.full(N * K, -1, np.int64)
    r = 0
    for e in range(E):
        for n in range(N):
            for k in range(K):
                if idx[n, k] == e:
                    row_map[n * K + k] = r
                    r += 1
    return row_map


def test_dispatch_golden():
    g = golden_dict("dispatch_small.txt")
    N, E, K = int(g["N"][0]), int(g["E"][0]), int(g["K"][0])
    idx = np.array(g["topk_idx"], np.int32).reshape(N, K)
    counts, offsets, row_map, src_slot = oracle.dispatch(idx, E)
    for key, val in (("counts", counts), ("offsets", offsets), ("row_map", row_map),
                     ("src_slot", src_slot)):
        assert np.array_equal(val, np.array(g[key], np.int32)), key


@pytest.mark.parametrize("N,E,K", [(1, 1, 1), (7, 3, 2), (50, 16, 4), (33, 8, 8), (200, 64, 2)])
def test_dispatch_brute_force_and_stable_argsort(N, E, K):
    idx = mi.random_topk_idx(N, E, K, seed=N + E + K).numpy()
    counts, offsets, row_map, src_slot = oracle.dispatch(idx, E)
    assert np.array_equal(row_map, brute_force_dispatch(idx, E))
    ref_src = np.argsort(idx.ravel(), kind="stable")
    assert np.array_equal(src_slot, ref_src)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))


def test_dispatch_invariants_100_seeds():
    # token conservation sum(counts) == N*K over 100 seeds (moe-engine page, Token守恒验证)
    for seed in range(100):
        X, W, _ = mi.make_route_inputs(64, 32, 8, seed)
        idx, _ = oracle.route(mi.bf16_bits(X), mi.bf16_bits(W), None, 2)
        counts, offsets, row_map, src_slot = oracle.dispatch(idx, 8)
        assert counts.sum() == 64 * 2
        assert offsets[-1] == 128 and np.all(np.diff(offsets) >= 0)
        assert np.array_equal(np.sort(row_map), np.arange(128))
        assert np.array_equal(src_slot[row_map], np.arange(128))
        assert all(len(set(r)) == 2 for r in idx)  # K distinct experts per token
        for e in range(8):
            slots = src_slot[offsets[e]:offsets[e + 1]]
            assert np.all(idx.ravel()[slots] == e)
            assert np.all(np.diff(slots // 2) > 0)  # tokens increase inside a range


def test_dispatch_empty_and_bad_index():
    c, o, r, s = oracle.dispatch(np.zeros((0, 2), np.int32), 4)
    assert np.all(c == 0) and np.all(o == 0) and r.size == 0
    with pytest.raises(oracle.OracleError):
        oracle.dispatch(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(oracle.OracleError):
        oracle.dispatch(np.array([[-1, 0]], np.int32), 4)


# ---------------------------------------------------------------- permute / E4M3

def test_permute_rows():
    N, H, E, K = 33, 40, 8, 3
    X = mi.random_bf16((N, H), seed=1)
    idx = mi.random_topk_idx(N, E, K, seed=2).numpy()
    _, _, row_map, _ = oracle.dispatch(idx, E)
    Xp = oracle.permute(mi.bf16_bits(X), row_map, K)
    ref = np.empty_like(Xp)
    ref[row_map] = np.repeat(mi.bf16_bits(X), K, axis=0)
    assert np.array_equal(Xp, ref)


def test_permute_fp8_matches_library_cast():
    N, H, E, K = 20, 384, 8, 2
    X = mi.random_bf16((N, H), seed=3, scale=3.0)
    X[0, :128] = 0.0                     # an all-zero block takes the clamped scale
    X[1, 128:256] *= 1e-6                # a tiny block
    X[2, 256:] *= 500.0                  # a large block
    idx = mi.random_topk_idx(N, E, K, seed=4).numpy()
    _, _, row_map, src_slot = oracle.dispatch(idx, E)
    Xp, Xq, Xs = oracle.permute(mi.bf16_bits(X), row_map, K, fp8=True)
    xs = X.to(torch.float32).numpy()
    for r in range(N * K):
        n = src_slot[r] // K
        for b in range(H // 128):
            blk = xs[n, b * 128:(b + 1) * 128]
            s = Xs[r, b]
            assert s == float(2.0 ** math.ceil(math.log2(
                float(np.float32(max(np.float32(np.abs(blk).max()), np.float32(1e-4)))
                      * np.float32(1 / 448)))))
            q_ref = torch.from_numpy((blk / s).astype(np.float32)).to(torch.float8_e4m3fn)
            assert np.array_equal(Xq[r, b * 128:(b + 1) * 128], q_ref.view(torch.uint8).numpy())
            # dequantised error is at most half an E4M3 step at that magnitude
            deq = torch.from_numpy(Xq[r, b * 128:(b + 1) * 128]).view(torch.float8_e4m3fn).double().numpy() * s
            step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(blk / s), 2.0**-6))) - 3), 2.0**-9) * s
            assert np.all(np.abs(deq - blk) <= 0.5 * step + 1e-30)
            assert np.all(np.abs(blk / s) <= 448.0)


# ---------------------------------------------------------------- combine

def test_combine_golden():
    g = golden_dict("combine_small.txt")
    N, H, K = int(g["N"][0]), int(g["H"][0]), int(g["K"][0])
    Y = to_bits([float(v) for v in g["Y"]]).reshape(N * K, H)
    w = np.array(g["w"], np.float32).reshape(N, K)
    out = oracle.combine(Y, np.array(g["row_map"], np.int32), w)
    assert np.array_equal(widen(out).ravel(), np.array(g["out"], np.float64))


def test_combine_matches_fp64_einsum_within_half_ulp():
    N, H, E, K = 40, 64, 8, 4
    Y = mi.random_bf16((N * K, H), seed=5)
    w = mi.random_weights(N, K, seed=6).numpy()
    idx = mi.random_topk_idx(N, E, K, seed=7).numpy()
    _, _, row_map, _ = oracle.dispatch(idx, E)
    out = widen(oracle.combine(mi.bf16_bits(Y), row_map, w))
    Yd = widen(mi.bf16_bits(Y))
    ref = np.einsum("nk,nkh->nh", w.astype(np.float64), Yd[row_map.reshape(N, K)])
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0**-126))) - 7)
    assert np.all(np.abs(out - ref) <= 0.5 * ulp)


def test_combine_residual_single_rounding():
    # forward_aggregate adds the residual before the one bf16 rounding:
    # 1 + 2^-8 + 2^-10 - 2^-9 = 1 + 0.375 ulp -> 1.0 (rounding the weighted sum
    # first would give 1 + 2^-7).  Second column: small integers and quarters,
    # exactly representable, so the result is the exact value.
    Y = to_bits([1.0, 3.0, 2.0 ** -8, -5.0, 2.0 ** -10, 7.0]).reshape(3, 2)
    w = np.array([[1.0, 1.0, 1.0]], np.float32)
    w2 = np.array([[0.5, 0.25, 1.0]], np.float32)
    R = to_bits([-(2.0 ** -9), 4.0]).reshape(1, 2)
    rm = np.array([0, 1, 2], np.int32)
    out = widen(oracle.combine_residual(Y, rm, w, R)).ravel()
    assert out[0] == 1.0
    assert out[1] == 3.0 - 5.0 + 7.0 + 4.0
    out2 = widen(oracle.combine_residual(Y, rm, w2, R)).ravel()
    assert out2[1] == 0.5 * 3.0 + 0.25 * -5.0 + 7.0 + 4.0


def test_combine_residual_matches_fp64_einsum_within_half_ulp():
    N, H, E, K = 40, 64, 8, 4
    Y = mi.random_bf16((N * K, H), seed=15)
    R = mi.random_bf16((N, H), seed=16, scale=3.0)
    w = mi.random_weights(N, K, seed=17).numpy()
    idx = mi.random_topk_idx(N, E, K, seed=18).numpy()
    _, _, row_map, _ = oracle.dispatch(idx, E)
    out = widen(oracle.combine_residual(mi.bf16_bits(Y), row_map, w, mi.bf16_bits(R)))
    Yd = widen(mi.bf16_bits(Y))
    ref = np.einsum("nk,nkh->nh", w.astype(np.float64), Yd[row_map.reshape(N, K)]) + widen(mi.bf16_bits(R))
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0**-126))) - 7)
    assert np.all(np.abs(out - ref) <= 0.5 * ulp)


def test_combine_residual_special_cases():
    N, H, E, K = 25, 32, 6, 3
    Y = mi.bf16_bits(mi.random_bf16((N * K, H), seed=19))
    R = mi.random_bf16((N, H), seed=20)
    R[R == 0] = 1.0                       # keep -0 out: 0 + (-0) is +0
    R = mi.bf16_bits(R)
    idx = mi.random_topk_idx(N, E, K, seed=21).numpy()
    _, _, row_map, _ = oracle.dispatch(idx, E)
    w = mi.random_weights(N, K, seed=22).numpy()
    # zero weights: the residual comes back bit for bit
    assert np.array_equal(oracle.combine_residual(Y, row_map, np.zeros_like(w), R), R)
    # zero residual: the plain weighted combine
    assert np.array_equal(oracle.combine_residual(Y, row_map, w, np.zeros_like(R)),
                          oracle.combine(Y, row_map, w))


def test_expert_fixture_matches_torch_fp32():
    rows, H, E = 30, 16, 5
    Xp = mi.random_bf16((rows, H), seed=8)
    counts = np.array([6, 0, 10, 4, 10], np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    Y = oracle.expert_fixture(mi.bf16_bits(Xp), offsets)
    expert = np.repeat(np.arange(E), counts)
    scale = torch.tensor([np.float32(1.0 + e / E) for e in expert], dtype=torch.float32)
    ref = (Xp.to(torch.float32) * scale[:, None]).to(torch.bfloat16)
    assert np.array_equal(Y, mi.bf16_bits(ref))


def test_whole_path_closed_form():
    # out[n] ~= X[n] * sum_k w_k (1 + e_k/E): every factor positive, no cancellation
    X, W, _ = mi.make_route_inputs(96, 64, 16, seed=9)
    r = oracle.run_path(mi.bf16_bits(X), mi.bf16_bits(W), None, 2)
    f = (r["topk_w"].astype(np.float64) * (1.0 + r["topk_idx"] / 16.0)).sum(axis=1)
    ref = widen(mi.bf16_bits(X)) * f[:, None]
    out = widen(r["out"])
    assert np.all(np.abs(out - ref) <= 1e-2 * np.abs(ref) + 1e-30)


def test_oracle_results_do_not_depend_on_thread_count():
    # the CPU baseline times the oracle on every host core and on one; the results are the same
    X, W, _ = mi.make_route_inputs(300, 128, 16, 7)
    Xb, Wb = mi.bf16_bits(X), mi.bf16_bits(W)
    n = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        assert oracle.num_threads() == 1 or n == 1
        one = oracle.run_path(Xb, Wb, None, 2)
    finally:
        oracle.set_num_threads(n)
    assert oracle.num_threads() == n
    many = oracle.run_path(Xb, Wb, None, 2)
    for key in ("topk_idx", "topk_w", "row_map", "Xp", "out"):
        assert np.array_equal(one[key], many[key]), key
