"""Comparison rules between the CUDA path and the CPU oracle.

Acceptance (from the statement of the routing problem, made precise):
  * top-K indices: identical, except at tokens where the oracle's fp64 logits
    of the swapped experts lie within NEAR_TIE (1e-3) of each other -- the
    fp32 tensor-core accumulation may order such experts differently.  A
    mismatching token is accepted only if the GPU picked K distinct experts,
    each with an oracle logit >= L_(K) - NEAR_TIE, in an order that never
    inverts two oracle logits by more than NEAR_TIE.  Counted and reported.
  * weights: within 1e-5 absolute of the oracle's weights for the same set;
  * dispatch metadata, permuted rows, E4M3 codes and scales: bit-exact when
    both sides are given the same indices;
  * combine: |gpu - ref| <= 1e-2 |ref| elementwise (bf16 output).
"""
from __future__ import annotations

import numpy as np

NEAR_TIE = 1e-3
W_ATOL = 1e-5
COMBINE_RTOL = 1e-2


def compare_topk(gpu_idx, gpu_w, ora_idx, ora_w, ora_logits, ora_probs=None, renorm=True):
    """Returns a dict of counts; raises AssertionError on an unacceptable mismatch."""
    gpu_idx = np.asarray(gpu_idx)
    gpu_w = np.asarray(gpu_w, dtype=np.float64)
    N, K = ora_idx.shape
    E = ora_logits.shape[1]
    same = np.all(gpu_idx == ora_idx, axis=1)
    # tokens in the near-tie zone: some adjacent gap among the top K+1 below NEAR_TIE
    srt = -np.sort(-ora_logits, axis=1)[:, :min(K + 1, E)]
    zone = np.any(np.abs(np.diff(srt, axis=1)) < NEAR_TIE, axis=1) if srt.shape[1] > 1 else np.zeros(N, bool)
    accepted = 0
    bad = []
    for n in np.nonzero(~same)[0]:
        g = gpu_idx[n]
        ok = (len(set(g.tolist())) == K and np.all((g >= 0) & (g < E)))
        if ok:
            Lg = ora_logits[n, g]
            kth = srt[n, K - 1]
            ok = bool(np.all(Lg >= kth - NEAR_TIE) and np.all(np.diff(Lg) <= NEAR_TIE))
        if ok:
            accepted += 1
        else:
            bad.append(int(n))
    assert not bad, (f"{len(bad)} tokens with top-K mismatches outside the near-tie rule, e.g. token "
                     f"{bad[0]}: gpu {gpu_idx[bad[0]].tolist()} oracle {ora_idx[bad[0]].tolist()} "
                     f"logits {ora_logits[bad[0], ora_idx[bad[0]]].tolist()}")
    # weights: where the sets agree, against the oracle's weights directly
    if np.any(same):
        err = np.max(np.abs(gpu_w[same] - ora_w[same].astype(np.float64)))
        assert err <= W_ATOL, f"weight error {err}"
    # where they differ (accepted near ties), against the oracle's probabilities of the GPU's set
    if accepted and ora_probs is not None:
        for n in np.nonzero(~same)[0]:
            p = ora_probs[n, gpu_idx[n]]
            ref = p / p.sum() if renorm else p
            assert np.max(np.abs(gpu_w[n] - ref)) <= W_ATOL
    return dict(tokens=int(N), mismatched=int((~same).sum()), near_tie_accepted=accepted,
                near_tie_zone=int(zone.sum()))


def check_dispatch_properties(idx, E, counts, offsets, row_map, src_slot):
    """Properties any correct dispatch of `idx` has (used where no oracle run exists)."""
    idx = np.asarray(idx)
    N, K = idx.shape
    S = N * K
    flat = idx.ravel()
    assert counts.sum() == S
    assert offsets[0] == 0 and offsets[-1] == S and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(row_map), np.arange(S))
    if src_slot is not None:
        assert np.array_equal(src_slot[row_map], np.arange(S))
    order = np.empty(S, np.int64)
    order[row_map] = np.arange(S)
    for e in range(E):
        sl = order[offsets[e]:offsets[e + 1]]
        assert np.all(flat[sl] == e)
        assert np.all(np.diff(sl) > 0)


def combine_close(gpu_bits, ref_bits, extra_atol=None):
    g = (np.asarray(gpu_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (np.asarray(ref_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    tol = COMBINE_RTOL * np.abs(r)
    if extra_atol is not None:
        tol = tol + extra_atol
    err = np.abs(g - r)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), f"combine mismatch at {worst}: gpu {g[worst]} ref {r[worst]}"
    return float(np.max(err / np.maximum(np.abs(r), 1e-30)))
