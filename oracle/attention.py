"""Decode attention over an int8-quantized KV cache (oracle).

What is computed, per query row (sequence b, draft column j, query head h):

  1. int8 query: (q8, qs) = per-head absmax/127 quantization of q[b, j, h]
     ("Kestrel_VLLM - 18", §3.3: int8 query quantization + int32 QK dot).
  2. kv head kh = h // g, g = Hq / Hkv (contiguous GQA groups).
  3. Column j attends to the first L_j = ctx[b] + j rows of sequence b, i.e.
     cache rows row_start[b] .. row_start[b] + L_j - 1 (draft column j sees
     the context plus drafts 0..j; "Kestrel_VLLM - 18", §二: batch column j
     must equal an M=1 decode that saw the same tokens).
  4. S_t = sum_i q8_i * k8_t,i exactly (int64 here; |S| <= 128*127^2).
  5. s_t = ((f32(S_t) * (qs * ks_t)) * sm_scale) in float32, sm_scale =
     RN_f32(1/sqrt(d)) unless given.  Parity unpinned: this order is the
     reading used here; the pages print no scaling order ("在 agent 时代如何
     快速验证 kernel 对精度的影响" writes only q @ K^T / sqrt(d)).
  6. softmax over t and the weighted sum of dequantized V rows
     vdeq_t = vs_t * v8_t.

Three ways to evaluate 6:

* ``reference`` with p_mode 0 -- the plain definition in float64:
      out = sum_t exp(s_t - max s) vdeq_t / sum_t exp(s_t - max s)
* ``reference`` with p_mode 1..5 -- the blockwise online softmax of
  "在 agent 时代如何快速验证 kernel 对精度的影响" (section "注意力权重"), with
  the rounding points placed where a split-KV kernel places them: keys are
  cut into splits of C keys (absolute positions [sC, (s+1)C)), each split
  into blocks of Bk keys; per block the running max m is updated first,
  p = f32(exp(s - m)) is rounded once to float32, the row sum uses p and the
  PV product uses round_p(p).  Splits are then merged in split order with
  weights exp(m_s - max_s m_s).  All other arithmetic is float64.  Mode 5
  multiplies the int8 V values by pv_operand(round_p(p), vs): the float32
  product p~ * vs rounded to 11 significant bits (rounding.py); mode 5 has
  no ``exact`` form.
* ``exact`` -- a float32 emulation of the sequential scan: one token at a
  time in token order, every float32 operation rounded on its own (no fused
  multiply-add), exp by the table-driven expf_tang:
      vdeq = f32(v8) * vs
      m'   = max(m, s_t)
      a    = expf_tang(m - m')          (m starts at -inf: a = 0)
      p    = expf_tang(s_t - m')
      l    = l * a + p
      o_i  = o_i * a + round_p(p) * vdeq_i
      m    = m'
  and out = o / l.  This is the operation order of the bit-exact scan in
  "Kestrel_VLLM - 18" §3.3 as read here (the page names the CPU function it
  mirrors but does not print it).
"""

from __future__ import annotations

import math
from decimal import Decimal, localcontext

import numpy as np

from .expf_tang import expf_tang
from .quant import quantize_queries
from .rounding import DIRECT, pv_operand, round_p, round_p_f32


def default_sm_scale(d: int) -> np.float32:
    """RN_f32(1/sqrt(d)), computed at 50 digits then rounded once to float32
    (the double from the decimal string is exact enough: float32 then rounds
    the 50-digit value's nearest double, which is not near a float32 tie)."""
    with localcontext() as ctx:
        ctx.prec = 50
        val = Decimal(1) / Decimal(d).sqrt()
    return np.float32(float(val))


def qk_int(q8_rows, k8_rows) -> np.ndarray:
    """Exact int64 dot products: q8_rows [R][d] x k8_rows [L][d] -> [R][L]."""
    return np.asarray(q8_rows, np.int64) @ np.asarray(k8_rows, np.int64).T


def scale_scores(S, qs, ks, sm_scale) -> np.ndarray:
    """s = ((f32(S) * (qs * ks)) * sm_scale), each product one f32 rounding.

    S [R][L] ints, qs [R] float32, ks [L] float32 -> float32 [R][L].
    """
    Sf = np.asarray(S).astype(np.float32)                    # exact: |S| < 2^24
    qk = np.multiply(np.asarray(qs, np.float32)[:, None],
                     np.asarray(ks, np.float32)[None, :], dtype=np.float32)
    s = np.multiply(Sf, qk, dtype=np.float32)
    return np.multiply(s, np.float32(sm_scale), dtype=np.float32)


# ---------------------------------------------------------------- per row --

def row_softmax_f64(s, vdeq) -> np.ndarray:
    """Plain softmax-weighted sum in float64."""
    s = np.asarray(s, np.float64)
    p = np.exp(s - s.max())
    return (p @ vdeq) / p.sum()


def row_online_mirrored(s, vdeq, p_mode: int, C: int, Bk: int, v8=None, vs=None) -> np.ndarray:
    """Blockwise online softmax with round_p, splits of C and blocks of Bk.

    vdeq [L][d] float64 = vs * v8; mode 5 (DIRECT) needs v8 [L][d] and vs [L]
    instead, since its PV operand is p~ * vs rounded."""
    s = np.asarray(s, np.float32)
    L = s.shape[0]
    parts = []
    for s0 in range(0, L, C):
        m, l, o = -math.inf, 0.0, np.zeros(vdeq.shape[1])
        for b0 in range(s0, min(s0 + C, L), Bk):
            b1 = min(b0 + Bk, s0 + C, L)
            sb = s[b0:b1].astype(np.float64)
            m_new = max(m, float(sb.max()))
            alpha = math.exp(m - m_new) if m != -math.inf else 0.0
            p = np.exp(sb - m_new).astype(np.float32)        # one f32 rounding
            l = l * alpha + float(p.astype(np.float64).sum())
            if p_mode == DIRECT:
                o = o * alpha + pv_operand(round_p(p, p_mode), vs[b0:b1], p_mode) @ \
                    np.asarray(v8[b0:b1], np.float64)
            else:
                o = o * alpha + round_p(p, p_mode) @ vdeq[b0:b1]
            m = m_new
        parts.append((m, l, o))
    m_all = max(pm for pm, _, _ in parts)
    l_tot, o_tot = 0.0, np.zeros(vdeq.shape[1])
    for pm, pl, po in parts:                                 # split order
        w = math.exp(pm - m_all)
        l_tot += w * pl
        o_tot = o_tot + w * po
    return o_tot / l_tot


def rows_exact_f32(s, v8, vs, p_mode: int) -> np.ndarray:
    """Sequential float32 scan for R rows sharing one key range.

    s [R][L] float32 scores; v8 [L][d] int8; vs [L] float32 -> out [R][d].
    Rows are independent; they are stepped together only to vectorise over
    rows and channels.  Each line is one float32 rounding per element.
    """
    s = np.asarray(s, np.float32)
    R, L = s.shape
    d = v8.shape[1]
    m = np.full(R, -np.inf, dtype=np.float32)
    l = np.zeros(R, dtype=np.float32)
    o = np.zeros((R, d), dtype=np.float32)
    for t in range(L):
        vdeq = np.multiply(v8[t].astype(np.float32), np.float32(vs[t]), dtype=np.float32)
        m_new = np.maximum(m, s[:, t])
        a = np.array([expf_tang(x) for x in np.subtract(m, m_new, dtype=np.float32)],
                     dtype=np.float32)
        p = np.array([expf_tang(x) for x in np.subtract(s[:, t], m_new, dtype=np.float32)],
                     dtype=np.float32)
        l = np.add(np.multiply(l, a, dtype=np.float32), p, dtype=np.float32)
        pr = round_p_f32(p, p_mode)
        o = np.add(np.multiply(o, a[:, None], dtype=np.float32),
                   np.multiply(pr[:, None], vdeq[None, :], dtype=np.float32),
                   dtype=np.float32)
        m = m_new
    return np.divide(o, l[:, None], dtype=np.float32)


# ------------------------------------------------------------- whole call --

def _check(q, k8, ks, v8, vs, row_start, ctx):
    B, M, Hq, d = q.shape
    Hkv = k8.shape[0]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    for b in range(B):
        if ctx[b] < 1 or row_start[b] < 0 or row_start[b] + ctx[b] + M - 1 > k8.shape[1]:
            raise ValueError(f"sequence {b} out of range")
    return B, M, Hq, Hkv, d


NO_SCORE = np.iinfo(np.int64).min   # cannot be a score: |S| <= 128 * 127^2


def qk_scores(q, k8, row_start, ctx):
    """Reference for the QK debug entry point.

    Returns (S int64 [B][M][Hq][max_ctx + M - 1] holding NO_SCORE where
    t >= L_j, q8 int8 [B][M][Hq][d], qs float32 [B][M][Hq]).
    """
    q = np.asarray(q, np.float32)
    B, M, Hq, Hkv, d = _check(q, k8, None, None, None, row_start, ctx)
    g = Hq // Hkv
    q8, qs = quantize_queries(q)
    width = int(np.max(ctx)) + M - 1
    S = np.full((B, M, Hq, width), NO_SCORE, dtype=np.int64)
    for b in range(B):
        for j in range(M):
            L = int(ctx[b]) + j
            r0 = int(row_start[b])
            for kh in range(Hkv):
                hs = slice(kh * g, (kh + 1) * g)
                S[b, j, hs, :L] = qk_int(q8[b, j, hs], k8[kh, r0:r0 + L])
    return S, q8, qs


def decode(q, k8, ks, v8, vs, row_start, ctx, *, sm_scale=None, p_mode=0,
           mode="reference", C=512, Bk=64, rows=None):
    """Decode attention for every (b, j, h), or for the listed ``rows``.

    q [B][M][Hq][d] float32; k8/v8 [Hkv][cap][d] int8; ks/vs [Hkv][cap]
    float32; row_start int64 [B]; ctx int32 [B] (>= 1).
    mode "reference" returns float64, mode "exact" returns float32.
    C, Bk place the rounding points of the rounded-P reference modes.
    rows: optional iterable of (b, j, h); other outputs are left NaN.
    """
    q = np.asarray(q, np.float32)
    B, M, Hq, Hkv, d = _check(q, k8, ks, v8, vs, row_start, ctx)
    g = Hq // Hkv
    sm = default_sm_scale(d) if sm_scale in (None, 0) else np.float32(sm_scale)
    q8, qs = quantize_queries(q)
    out = np.full(q.shape, np.nan, dtype=np.float64 if mode == "reference" else np.float32)
    want = None if rows is None else {}
    if rows is not None:
        for (b, j, h) in rows:
            want.setdefault((b, j), set()).add(h)
    for b in range(B):
        r0 = int(row_start[b])
        for j in range(M):
            if want is not None and (b, j) not in want:
                continue
            L = int(ctx[b]) + j
            heads = range(Hq) if want is None else sorted(want[(b, j)])
            for kh in range(Hkv):
                hs = [h for h in heads if h // g == kh]
                if not hs:
                    continue
                kr, vr = k8[kh, r0:r0 + L], v8[kh, r0:r0 + L]
                S = qk_int(q8[b, j, hs], kr)
                s = scale_scores(S, qs[b, j, hs], ks[kh, r0:r0 + L], sm)
                if mode == "exact":
                    out[b, j, hs] = rows_exact_f32(s, vr, vs[kh, r0:r0 + L], p_mode)
                    continue
                vdeq = vs[kh, r0:r0 + L].astype(np.float64)[:, None] * vr.astype(np.float64)
                for i, h in enumerate(hs):
                    if p_mode == 0:
                        out[b, j, h] = row_softmax_f64(s[i], vdeq)
                    else:
                        out[b, j, h] = row_online_mirrored(s[i], vdeq, p_mode, C, Bk,
                                                           v8=vr, vs=vs[kh, r0:r0 + L])
    return out
