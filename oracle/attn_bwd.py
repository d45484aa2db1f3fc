"""fp64 CPU oracle for the Ring Attention backward step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use
it; the GPU library never does.

The mKernel pages do not describe the backward step; it is the gradient of the forward
step they do describe (oracle.c: softmax(scale * Q K^T [+ causal mask over global
positions]) V, with the per-row log-sum-exp).  For one (b, hq) with kv = hq / (Hq/Hkv),
scores s_ij = scale * q_i . k_j over the allowed keys A_i, P = softmax_j(s), O = P V and an
upstream gradient dO, the chain rule gives

    dV_j  = sum_i P_ij dO_i                                  (summed over the query heads
    dP_ij = dO_i . v_j                                        that share the KV head)
    D_i   = dO_i . O_i             ( = sum_j P_ij dP_ij )
    dS_ij = P_ij (dP_ij - D_i)
    dQ_i  = scale * sum_j dS_ij k_j
    dK_j  = scale * sum_i dS_ij q_i                          (summed like dV)

in fp64 from the bf16 inputs, with P, O and D taken from this module's own fp64 forward
(not from any GPU output).  The ring order in which the chunks are visited does not change
these sums.  The matrix products are numpy float64 matmuls, library primitives used as steps.

Parity status: pinned (tests/test_oracle_attn_bwd.py): central finite differences of the
forward oracle (oracle.c, itself pinned) along random directions, the single-key and
uniform-attention closed forms, GQA as a sum over repeated heads, and a mutation check.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _scores(qh, kh, scale, causal, q0=0):
    """scale * Q K^T for query rows q0 .. q0+len(qh)-1, -inf where the causal mask forbids."""
    s = scale * (qh @ kh.T)
    if causal:
        qi = np.arange(q0, q0 + qh.shape[0])[:, None]
        kj = np.arange(kh.shape[0])[None, :]
        s = np.where(kj > qi, -np.inf, s)
    return s


def _softmax(s):
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def attn_bwd(q_bits, k_bits, v_bits, do_bits, *, causal, scale=None):
    """Full gradients.  q, do: [B][Hq][S][d]; k, v: [B][Hkv][S][d] (bf16 bits).
    Returns (dq [B][Hq][S][d], dk [B][Hkv][S][d], dv [B][Hkv][S][d]) in float64."""
    q, k, v, do = (bf16_to_f64(x) for x in (q_bits, k_bits, v_bits, do_bits))
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            s = _scores(q[b, h], k[b, kv], scale, causal)
            p, _ = _softmax(s)
            o = p @ v[b, kv]
            dv[b, kv] += p.T @ do[b, h]
            dp = do[b, h] @ v[b, kv].T
            D = np.sum(do[b, h] * o, axis=1)
            ds = p * (dp - D[:, None])
            dq[b, h] = scale * (ds @ k[b, kv])
            dk[b, kv] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def lse_and_delta(q_bits, k_bits, v_bits, do_bits, b, h, Hq, Hkv, *, causal, scale, block=1024, with_ed=False):
    """LSE_i (natural log) and D_i = dO_i . O_i for every query row of head (b, h), in
    blocks of query rows (the full-size checks need them for every row).  with_ed: also eD_i
    and vD_i of error_scales."""
    q, k, v, do = (bf16_to_f64(x) for x in (q_bits[b, h], k_bits[b, h // (Hq // Hkv)],
                                              v_bits[b, h // (Hq // Hkv)], do_bits[b, h]))
    S = q.shape[0]
    lse = np.empty(S)
    D = np.empty(S)
    ed = np.empty(S)
    vd = np.empty(S)
    for i0 in range(0, S, block):
        s = _scores(q[i0:i0 + block], k, scale, causal, q0=i0)
        p, l = _softmax(s)
        lse[i0:i0 + block] = l
        o = p @ v
        D[i0:i0 + block] = np.sum(do[i0:i0 + block] * o, axis=1)
        if with_ed:
            dob = do[i0:i0 + block]
            ed[i0:i0 + block] = np.sum(np.abs(dob) * (np.abs(o) + p @ np.abs(v)), axis=1)
            vd[i0:i0 + block] = np.sum(dob ** 2 * (o ** 2 + (p ** 2) @ (v ** 2)), axis=1)
    return (lse, D, ed, vd) if with_ed else (lse, D)


def error_scales(q_bits, k_bits, v_bits, do_bits, *, causal, scale=None):
    """Magnitudes that bound what a bf16 implementation's roundings do to the gradients (test
    tolerance, not a gradient).  The path modelled takes O in bf16 from a forward that rounded P
    to bf16 before P V, rounds P to bf16 before P dO and before forming dS, rounds dS to bf16
    before dS K and dS^T Q, rounds each gradient to bf16, and accumulates in fp32.  With u the
    relative rounding error of bf16 (|eps| <= u for each rounding), each gradient element
    G = sum_t (term t) deviates by sum_t eps_t (term t) over the rounding sites, plus at most
    u |G| for its own rounding and the fp32 accumulation error.

    Worst case (signs aligned), to first order in u: |dG| <= u (E + |G|), where

        eD_i  = sum_c |dO_ic| (|O_ic| + sum_j P_ij |v_jc|)       (|error of D_i| <= u eD_i)
        Ev_jc = sum_i P_ij |dO_ic|
        Ek_jc = scale sum_i (2 |dS_ij| + P_ij eD_i) |q_ic|      (dS: the roundings of P and of
        Eq_ic = scale sum_j (2 |dS_ij| + P_ij eD_i) |k_jc|       dS, and D's error times P)

    Independent roundings (zero mean, variance <= u^2 / 3 each): E ||dG||^2 <= (u^2 / 3) sum T2
    (plus the gradients' own rounding), with per-element sums of squared terms

        vD_i  = sum_c dO_ic^2 (O_ic^2 + sum_j P_ij^2 v_jc^2)
        T2v_jc = sum_i P_ij^2 dO_ic^2
        T2k_jc = scale^2 sum_i (2 dS_ij^2 + P_ij^2 vD_i) q_ic^2
        T2q_ic = scale^2 sum_j (2 dS_ij^2 + P_ij^2 vD_i) k_jc^2

    All summed over the query heads that share a KV head, like the gradients.  Returns
    ((Eq, Ek, Ev), (T2q, T2k, T2v)) with the gradients' shapes."""
    q, k, v, do = (bf16_to_f64(x) for x in (q_bits, k_bits, v_bits, do_bits))
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    eq, tq = np.zeros_like(q), np.zeros_like(q)
    ek, tk = np.zeros_like(k), np.zeros_like(k)
    ev, tv = np.zeros_like(v), np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            kh, vh, qh, doh = k[b, kv], v[b, kv], q[b, h], do[b, h]
            p, _ = _softmax(_scores(qh, kh, scale, causal))
            o = p @ vh
            D = np.sum(doh * o, axis=1)
            ed = np.sum(np.abs(doh) * (np.abs(o) + p @ np.abs(vh)), axis=1)
            vd = np.sum(doh ** 2 * (o ** 2 + (p ** 2) @ (vh ** 2)), axis=1)
            ds = p * (doh @ vh.T - D[:, None])
            w1 = 2.0 * np.abs(ds) + p * ed[:, None]
            w2 = 2.0 * ds ** 2 + p ** 2 * vd[:, None]
            ev[b, kv] += p.T @ np.abs(doh)
            tv[b, kv] += (p ** 2).T @ (doh ** 2)
            ek[b, kv] += scale * (w1.T @ np.abs(qh))
            tk[b, kv] += scale ** 2 * (w2.T @ (qh ** 2))
            eq[b, h] = scale * (w1 @ np.abs(kh))
            tq[b, h] = scale ** 2 * (w2 @ (kh ** 2))
    return (eq, ek, ev), (tq, tk, tv)


def attn_bwd_rows(q_bits, k_bits, v_bits, do_bits, *, causal, scale, bh_rows, kv_rows, with_scales=False):
    """Sampled gradient rows.  bh_rows: flat query-row ids ((b*Hq + hq)*S + i) -> dQ rows;
    kv_rows: flat KV-row ids ((b*Hkv + kvh)*S + j) -> dK, dV rows (summed over the group's
    query heads).  Returns (dq [len(bh_rows)][d], dk, dv [len(kv_rows)][d]); with_scales: then
    ((dq, dk, dv), (eq, ek, ev), (t2q, t2k, t2v)), the rows of error_scales as well."""
    B, Hq, S, d = q_bits.shape
    Hkv = k_bits.shape[1]
    g = Hq // Hkv
    heads = sorted({int(r) // S for r in bh_rows} | {(int(r) // S // Hkv) * Hq + (int(r) // S % Hkv) * g + i
                                                      for r in kv_rows for i in range(g)})
    stats = {bh: lse_and_delta(q_bits, k_bits, v_bits, do_bits, bh // Hq, bh % Hq, Hq, Hkv, causal=causal,
                               scale=scale, with_ed=True) for bh in heads}
    q, k, v, do = (bf16_to_f64(x) for x in (q_bits, k_bits, v_bits, do_bits))
    dq, eq, tq = (np.zeros((len(bh_rows), d)) for _ in range(3))
    for n, r in enumerate(bh_rows):
        bh, i = int(r) // S, int(r) % S
        b, h = bh // Hq, bh % Hq
        kv = h // g
        lse, D, ed, vd = stats[bh]
        kk = k[b, kv, :i + 1] if causal else k[b, kv]
        vv = v[b, kv, :i + 1] if causal else v[b, kv]
        p = np.exp(scale * (kk @ q[b, h, i]) - lse[i])
        ds = p * (vv @ do[b, h, i] - D[i])
        dq[n] = scale * (ds @ kk)
        eq[n] = scale * ((2.0 * np.abs(ds) + p * ed[i]) @ np.abs(kk))
        tq[n] = scale ** 2 * ((2.0 * ds ** 2 + p ** 2 * vd[i]) @ (kk ** 2))
    dk, dv, ek, ev, tk, tv = (np.zeros((len(kv_rows), d)) for _ in range(6))
    for n, r in enumerate(kv_rows):
        bkv, j = int(r) // S, int(r) % S
        b, kv = bkv // Hkv, bkv % Hkv
        for h in range(kv * g, (kv + 1) * g):
            lse, D, ed, vd = stats[b * Hq + h]
            i0 = j if causal else 0
            qq, dd = q[b, h, i0:], do[b, h, i0:]
            p = np.exp(scale * (qq @ k[b, kv, j]) - lse[i0:])
            dv[n] += p @ dd
            ds = p * (dd @ v[b, kv, j] - D[i0:])
            dk[n] += scale * (ds @ qq)
            ev[n] += p @ np.abs(dd)
            tv[n] += (p ** 2) @ (dd ** 2)
            ek[n] += scale * ((2.0 * np.abs(ds) + p * ed[i0:]) @ np.abs(qq))
            tk[n] += scale ** 2 * ((2.0 * ds ** 2 + p ** 2 * vd[i0:]) @ (qq ** 2))
    if with_scales:
        return (dq, dk, dv), (eq, ek, ev), (tq, tk, tv)
    return dq, dk, dv


def attn_bwd_dq_rows(q_bits, k_bits, v_bits, do_bits, *, causal, scale, bh_rows):
    """dQ rows only, each from its own row of the forward (its LSE and D need no other
    query row).  bh_rows: flat query-row ids ((b*Hq + hq)*S + i).  Returns [len][d]."""
    B, Hq, S, d = q_bits.shape
    g = Hq // k_bits.shape[1]
    out = np.zeros((len(bh_rows), d))
    for n, r in enumerate(bh_rows):
        bh, i = int(r) // S, int(r) % S
        b, h = bh // Hq, bh % Hq
        n_keys = i + 1 if causal else S
        kk = bf16_to_f64(k_bits[b, h // g, :n_keys])
        vv = bf16_to_f64(v_bits[b, h // g, :n_keys])
        qi = bf16_to_f64(q_bits[b, h, i])
        doi = bf16_to_f64(do_bits[b, h, i])
        s = scale * (kk @ qi)
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        p = e / l
        D = doi @ (p @ vv)
        ds = p * (vv @ doi - D)
        out[n] = scale * (ds @ kk)
    return out


def for_workload(w, q, k, v, do):
    return attn_bwd(q, k, v, do, causal=bool(w.causal), scale=w.scale)
