"""Pins for the fp64 oracle: checks that tie it to something other than itself.

The pages print no worked numerical example, so the oracle is pinned by
what the mathematics of the method fixes:

  normalisation   softmax rows sum to one; masked entries are exactly zero
                  ("提示词再优…" §2.2 stable_softmax; causal flag, 第一章)
  identical_keys  closed form: equal keys give O = mean of the visible V
                  rows and lse = scale*q.k + ln(#visible)
  online          the one-pass running-max form of "Gemini 3 Flash的注意力内核
                  重写…" §3 在线softmax算法 equals the three-step form of
                  §传统注意力计算的内存带宽瓶颈
  causal_row0     causal row 0 sees only key 0: O_0 = V_0, lse_0 = s_00
  finite_diff     gradients equal central finite differences of L = sum(dO*O)
  invariants      key permutation, constant key shift (with very large
                  logits), sum_j dK_j = 0, sum_j dV_j = sum_i dO_i,
                  identical keys give dQ = 0
  zero_query      Q = 0 gives uniform attention: lse_i = ln(#visible)
  torch_sdpa      an independent library routine (PyTorch's fp64 CPU
                  scaled_dot_product_attention and autograd) agrees

Each pin is a function of an oracle object (``oracle.OracleLib``) so the same
checks also run against deliberately broken copies of the oracle source
(tests/test_oracle_mutants.py) to show that every plausible mistake is
caught by at least one of them.
"""
from __future__ import annotations

import numpy as np


def _rng(seed):
    return np.random.default_rng(seed)


def pin_normalisation(orc):
    """With V = identity rows, O_i is exactly the probability row p_i."""
    rng = _rng(11)
    for causal in (False, True):
        for N in (1, 5, 8):
            d = 8
            q = rng.standard_normal((N, d))
            k = rng.standard_normal((N, d))
            v = np.eye(N, d)
            o, lse = orc.head_fwd(q, k, v, causal, 0.7, nthreads=2)
            p = o[:, :N]
            assert np.all(np.isfinite(p))
            assert np.all(p >= 0.0)
            assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12
            if causal:
                assert np.all(p[np.triu_indices(N, 1)] == 0.0)
                assert np.all(p[np.tril_indices(N)] > 0.0)


def pin_identical_keys(orc):
    rng = _rng(12)
    N, d, scale = 13, 6, 0.4
    q = rng.standard_normal((N, d))
    kk = rng.standard_normal(d)
    k = np.tile(kk, (N, 1))
    v = rng.standard_normal((N, d))
    dO = rng.standard_normal((N, d))
    for causal in (False, True):
        o, lse = orc.head_fwd(q, k, v, causal, scale, nthreads=3)
        cnt = np.arange(1, N + 1) if causal else np.full(N, N)
        if causal:
            want_o = np.cumsum(v, axis=0) / cnt[:, None]
        else:
            want_o = np.tile(v.mean(axis=0), (N, 1))
        want_lse = scale * (q @ kk) + np.log(cnt)
        assert np.max(np.abs(o - want_o)) <= 1e-12
        assert np.max(np.abs(lse - want_lse)) <= 1e-12
        # equal keys: every row of dS sums against a single key -> dQ = 0
        dq, dk, dv = orc.head_bwd(q, k, v, dO, causal, scale, nthreads=3)
        assert np.max(np.abs(dq)) <= 1e-12


def pin_online(orc):
    rng = _rng(13)
    for N in (1, 7, 33, 64):
        for d in (4, 16):
            for sigma, scale in ((1.0, 0.5), (2.0, 0.25), (8.0, 1.0)):
                q = sigma * rng.standard_normal((N, d))
                k = sigma * rng.standard_normal((N, d))
                v = rng.standard_normal((N, d))
                for causal in (False, True):
                    o2, l2 = orc.head_fwd(q, k, v, causal, scale, nthreads=2)
                    for tile in (1, 3, 16):
                        o1, l1 = orc.head_fwd_online(q, k, v, causal, scale, tile)
                        assert np.max(np.abs(o1 - o2)) <= 1e-12, (N, d, sigma, causal, tile)
                        assert np.max(np.abs(l1 - l2)) <= 1e-12 * max(1.0, np.max(np.abs(l2)))


def pin_causal_row0(orc):
    rng = _rng(14)
    for N in (1, 4, 17):
        d = 5
        q = 3 * rng.standard_normal((N, d))
        k = 3 * rng.standard_normal((N, d))
        v = rng.standard_normal((N, d))
        o, lse = orc.head_fwd(q, k, v, True, 0.9, rows=[0], nthreads=1)
        assert np.array_equal(o[0], v[0])
        s00 = 0.9 * float(np.dot(q[0], k[0]))
        assert abs(lse[0] - s00) <= 1e-13 * max(1.0, abs(s00))


def _loss(orc, q, k, v, dO, causal, scale):
    o, _ = orc.head_fwd(q, k, v, causal, scale, nthreads=1)
    return float(np.sum(dO * o))


def pin_finite_diff(orc):
    rng = _rng(15)
    h = 1e-6
    for N, d in ((5, 4), (16, 8)):
        for causal in (False, True):
            scale = 1.0 / np.sqrt(d)
            q, k, v, dO = (rng.standard_normal((N, d)) for _ in range(4))
            dq, dk, dv = orc.head_bwd(q, k, v, dO, causal, scale, nthreads=2)
            for which, analytic in ((0, dq), (1, dk), (2, dv)):
                num = np.zeros((N, d))
                for i in range(N):
                    for c in range(d):
                        args_p = [q.copy(), k.copy(), v.copy()]
                        args_m = [q.copy(), k.copy(), v.copy()]
                        args_p[which][i, c] += h
                        args_m[which][i, c] -= h
                        num[i, c] = (_loss(orc, *args_p, dO, causal, scale)
                                     - _loss(orc, *args_m, dO, causal, scale)) / (2 * h)
                rel = np.linalg.norm(analytic - num) / max(np.linalg.norm(num), 1e-30)
                assert rel <= 1e-6, (N, d, causal, which, rel)


def pin_invariants(orc):
    rng = _rng(16)
    N, d = 24, 8
    scale = 1.0 / np.sqrt(d)
    q, k, v, dO = (rng.standard_normal((N, d)) for _ in range(4))
    # key/value permutation leaves O unchanged (non-causal)
    perm = rng.permutation(N)
    o, lse = orc.head_fwd(q, k, v, False, scale, nthreads=2)
    o_p, lse_p = orc.head_fwd(q, k[perm], v[perm], False, scale, nthreads=2)
    assert np.max(np.abs(o - o_p)) <= 1e-12
    assert np.max(np.abs(lse - lse_p)) <= 1e-12
    # constant shift of every key: O unchanged, lse shifts by scale*q.c; the
    # shift is large enough that exp of an unshifted logit overflows fp64
    for causal in (False, True):
        o0, l0 = orc.head_fwd(q, k, v, causal, scale, nthreads=2)
        c = 400.0 * rng.standard_normal(d)
        o1, l1 = orc.head_fwd(q, k + c, v, causal, scale, nthreads=2)
        assert np.all(np.isfinite(o1)) and np.all(np.isfinite(l1))
        assert np.max(np.abs(o1 - o0)) <= 1e-9
        assert np.max(np.abs((l1 - l0) - scale * (q @ c))) <= 1e-9 * np.max(np.abs(l1))
        # gradient sums
        dq, dk, dv = orc.head_bwd(q, k, v, dO, causal, scale, nthreads=2)
        assert np.max(np.abs(dk.sum(axis=0))) <= 1e-12
        assert np.max(np.abs(dv.sum(axis=0) - dO.sum(axis=0))) <= 1e-12
    # sampled rows/columns equal the same entries of the full evaluation
    for causal in (False, True):
        dq, dk, dv, lse_b, D = orc.head_bwd(q, k, v, dO, causal, scale, nthreads=2,
                                            want_stats=True)
        rows = [0, 5, N - 1]
        dq_s, dk_s, dv_s = orc.head_bwd(q, k, v, dO, causal, scale, qrows=rows, krows=rows,
                                        nthreads=1)
        assert np.array_equal(dq_s, dq[rows]) and np.array_equal(dk_s, dk[rows])
        assert np.array_equal(dv_s, dv[rows])
        o, lse = orc.head_fwd(q, k, v, causal, scale, nthreads=2)
        assert np.array_equal(lse, lse_b)
        assert np.max(np.abs(D - np.sum(dO * o, axis=1))) <= 1e-12


def pin_zero_query(orc):
    rng = _rng(17)
    N, d = 9, 4
    q = np.zeros((N, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    for causal in (False, True):
        o, lse = orc.head_fwd(q, k, v, causal, 0.5, nthreads=2)
        cnt = np.arange(1, N + 1) if causal else np.full(N, N)
        assert np.max(np.abs(lse - np.log(cnt))) <= 1e-13


def pin_torch_sdpa(orc, shapes=((1, 2, 256, 64, False), (1, 2, 160, 128, True))):
    import torch
    import torch.nn.functional as F
    for (B, H, N, d, causal) in shapes:
        g = torch.Generator().manual_seed(1234 + N)
        q, k, v, dO = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
        scale = 1.0 / np.sqrt(d)
        qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
        ot = F.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
        ot.backward(dO)
        o, lse = orc.attention_fwd(q.numpy(), k.numpy(), v.numpy(), causal, scale, nthreads=4)
        dq, dk, dv = orc.attention_bwd(q.numpy(), k.numpy(), v.numpy(), dO.numpy(), causal,
                                       scale, nthreads=4)
        assert np.max(np.abs(o - ot.detach().numpy())) <= 1e-12
        for mine, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
            assert np.max(np.abs(mine - ref.numpy())) <= 1e-11


def _window_counts(N, W, causal):
    """Visible keys per row under window W (closed form of the reading: i - j < W,
    and j - i < W when not causal)."""
    i = np.arange(N)
    lo = np.maximum(0, i - W + 1)
    hi = i if causal else np.minimum(N - 1, i + W - 1)
    return lo, hi, hi - lo + 1


def pin_window_identical_keys(orc):
    """Sliding window, identical keys: every visible score of a row is equal, so
    o_i is the mean of v over exactly the visible keys and lse_i adds ln(count)."""
    rng = _rng(21)
    N, d, scale = 23, 5, 0.7
    q = rng.standard_normal((N, d))
    kk = rng.standard_normal(d)
    k = np.tile(kk, (N, 1))
    v = rng.standard_normal((N, d))
    dO = rng.standard_normal((N, d))
    for causal in (True, False):
        for W in (1, 2, 5, 22, 23, 40):
            o, lse = orc.head_fwd(q, k, v, causal, scale, nthreads=3, window=W)
            lo, hi, cnt = _window_counts(N, W, causal)
            want_o = np.stack([v[lo[i]:hi[i] + 1].mean(axis=0) for i in range(N)])
            assert np.max(np.abs(o - want_o)) <= 1e-12, (causal, W)
            assert np.max(np.abs(lse - (scale * (q @ kk) + np.log(cnt)))) <= 1e-12, (causal, W)
            dq, dk, dv = orc.head_bwd(q, k, v, dO, causal, scale, nthreads=3, window=W)
            assert np.max(np.abs(dq)) <= 1e-12
            # dV_j = sum over the rows that see key j of p_ij dO_i, p_ij = 1/count_i
            want_dv = np.zeros((N, d))
            for i in range(N):
                want_dv[lo[i]:hi[i] + 1] += dO[i] / cnt[i]
            assert np.max(np.abs(dv - want_dv)) <= 1e-12, (causal, W)


def pin_window_one(orc):
    """Causal window 1: each row sees only its own key, so o_i = v_i exactly and
    lse_i = s_ii; a window of N or more is no window at all."""
    rng = _rng(22)
    N, d, scale = 17, 6, 0.45
    q, k, v = (2 * rng.standard_normal((N, d)) for _ in range(3))
    o, lse = orc.head_fwd(q, k, v, True, scale, nthreads=2, window=1)
    assert np.array_equal(o, v)
    sii = scale * np.einsum("ij,ij->i", q, k)
    assert np.max(np.abs(lse - sii)) <= 1e-13 * max(1.0, np.max(np.abs(sii)))
    for causal in (True, False):
        o0, l0 = orc.head_fwd(q, k, v, causal, scale, nthreads=2)
        oN, lN = orc.head_fwd(q, k, v, causal, scale, nthreads=2, window=N)
        assert np.array_equal(o0, oN) and np.array_equal(l0, lN)


def pin_window_online_and_fd(orc):
    """With a window, the one-pass tiled forward equals the three-step one, and
    the analytic gradient matches central finite differences."""
    rng = _rng(23)
    for N, d, W in ((9, 4, 3), (16, 8, 5)):
        scale = 1.0 / np.sqrt(d)
        q, k, v, dO = (rng.standard_normal((N, d)) for _ in range(4))
        for causal in (True, False):
            o2, l2 = orc.head_fwd(q, k, v, causal, scale, nthreads=2, window=W)
            for tile in (1, 3, 16):
                o1, l1 = orc.head_fwd_online(q, k, v, causal, scale, tile, window=W)
                assert np.max(np.abs(o1 - o2)) <= 1e-12 and np.max(np.abs(l1 - l2)) <= 1e-12
            dq, dk, dv = orc.head_bwd(q, k, v, dO, causal, scale, nthreads=2, window=W)
            h = 1e-6
            for which, analytic in ((0, dq), (1, dk), (2, dv)):
                num = np.zeros((N, d))
                for i in range(N):
                    for c in range(d):
                        ap = [q.copy(), k.copy(), v.copy()]
                        am = [q.copy(), k.copy(), v.copy()]
                        ap[which][i, c] += h
                        am[which][i, c] -= h
                        fp = float(np.sum(dO * orc.head_fwd(*ap, causal, scale, nthreads=1, window=W)[0]))
                        fm = float(np.sum(dO * orc.head_fwd(*am, causal, scale, nthreads=1, window=W)[0]))
                        num[i, c] = (fp - fm) / (2 * h)
                rel = np.linalg.norm(analytic - num) / max(np.linalg.norm(num), 1e-30)
                assert rel <= 1e-6, (N, d, W, causal, which, rel)


ALL_PINS = [pin_normalisation, pin_identical_keys, pin_online, pin_causal_row0, pin_finite_diff,
            pin_invariants, pin_zero_query, pin_torch_sdpa, pin_window_identical_keys, pin_window_one,
            pin_window_online_and_fd]
