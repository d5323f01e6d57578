"""Tie-aware comparison of the GPU router gating with the oracle's.

The oracle ranks in float64; the GPU ranks fp32 scores.  For the softmax
router both rank the same numbers (the fp32 logits: softmax is monotone), so
ids must match exactly.  For the sigmoid router the fp32 scores carry a few
ulps of error, so a token whose decision margins (group boundary, expert
boundary) exceed DELTA, or are exact ties (decided by the lower index on both
sides), must match the oracle exactly; a token with a closer call must give a
valid answer at that tolerance.
"""
import numpy as np

import oracle

# |fp32 score - exact score| <= a few ulps of values below ~2: s = sigmoid via
# expf (2 ulp) and one IEEE division, plus the bias, and group sums of two.
DELTA = 4e-6
WEIGHT_RTOL = 1e-5


def check_softmax(lg, k, ids, w, shared=False):
    E = lg.shape[1]
    ids_o, w_o = oracle.gate_softmax_topk(lg, k)
    np.testing.assert_array_equal(ids[:, :k], ids_o)
    np.testing.assert_allclose(w[:, :k], w_o, rtol=WEIGHT_RTOL, atol=1e-30)
    _check_shared(ids, w, k, E, shared)


def _check_shared(ids, w, k, E, shared):
    if shared:
        assert ids.shape[1] == k + 1
        assert (ids[:, k] == E).all() and (w[:, k] == 1.0).all()
    else:
        assert ids.shape[1] == k


def check_grouped(lg, k, n_group, topk_group, scale, bias, ids, w, shared=False, max_near_frac=0.01):
    """Returns the number of tokens that were only checked for validity."""
    M, E = lg.shape
    gs = E // n_group
    bias = np.zeros(E) if bias is None else np.asarray(bias, dtype=np.float64)
    ids_o, w_o = oracle.gate_grouped_sigmoid_topk(lg, k, n_group, topk_group, bias=bias, routed_scaling=scale)
    s = 1.0 / (1.0 + np.exp(-lg.astype(np.float64)))
    b = s + bias[None, :]
    gi, gw = ids[:, :k], w[:, :k]
    assert ((gi >= 0) & (gi < E)).all()
    near = 0
    for t in range(M):
        assert len(set(gi[t].tolist())) == k, f"token {t}: repeated ids {gi[t]}"
        grouped = b[t].reshape(n_group, gs)
        gscore = -np.sort(-grouped, axis=1)[:, :2].sum(axis=1) if gs >= 2 else grouped[:, 0]
        gsorted = np.sort(gscore)[::-1]
        g_margin = gsorted[topk_group - 1] - gsorted[topk_group] if topk_group < n_group else np.inf
        kept = set(np.argsort(-gscore, kind="stable")[:topk_group].tolist())
        cand = np.sort(np.concatenate([b[t, g * gs:(g + 1) * gs] for g in sorted(kept)]))[::-1]
        e_margin = cand[k - 1] - cand[k] if len(cand) > k else np.inf
        # an exact tie (gap 0) is decided by index on both sides; a gap within fp32 error is not
        if not (0 < g_margin <= DELTA or 0 < e_margin <= DELTA):
            assert set(gi[t].tolist()) == set(ids_o[t].tolist()), f"token {t}: {gi[t]} vs {ids_o[t]}"
            for j in range(k):  # column order: only near-equal scores may swap
                if gi[t, j] != ids_o[t, j]:
                    assert abs(b[t, gi[t, j]] - b[t, ids_o[t, j]]) <= DELTA, f"token {t} column {j}"
            pos = {int(e): j for j, e in enumerate(ids_o[t])}
            want = np.array([w_o[t, pos[int(e)]] for e in gi[t]])
            np.testing.assert_allclose(gw[t], want, rtol=WEIGHT_RTOL, atol=1e-30)
        else:
            near += 1
            groups = {int(e) // gs for e in gi[t]}
            assert len(groups) <= topk_group
            for g in groups:
                assert gscore[g] >= gsorted[topk_group - 1] - DELTA, f"token {t}: group {g} not among the best"
            chosen = set(gi[t].tolist())
            worst = min(b[t, e] for e in chosen)
            for g in groups:
                for e in range(g * gs, (g + 1) * gs):
                    if e not in chosen:
                        assert b[t, e] <= worst + DELTA, f"token {t}: expert {e} beats a chosen one"
            ss = s[t, gi[t]]
            np.testing.assert_allclose(gw[t], ss / ss.sum() * scale, rtol=WEIGHT_RTOL, atol=1e-30)
    assert near <= max(1, max_near_frac * M), f"{near} of {M} tokens had near-tied decisions"
    _check_shared(ids, w, k, E, shared)
    return near
