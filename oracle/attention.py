"""Absorbed MLA decode and its expanded reference (oracle; test infrastructure).

Sources (page title, section):

* "DeepSeek的MLA技术：极致压缩KV Cache的创新方案" (the juejin tutorial):
  "步骤2：从潜在空间生成各头的K、V" (K_i = C^KV W_i^upK, V_i = C^KV W_i^upV),
  the listing "完整的MLA注意力计算" (per-head softmax(Q K^T / sqrt(d)) V, then
  concatenation and W_o), and "KV Cache的实现" (append the latent, re-expand
  K/V for every cached token at each step).
* "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite — Technical Report",
  §1.3 (expanded K is 192 wide = nope 128 + rope 64, V is 128 wide, k_pe is
  shared by the heads) and §2.1 (the cache keeps compressed_kv [seq, 512]
  plus k_pe [seq, 64] and projects at compute time).

What is computed here, per sequence and head h, in fp64 over fp32 operands:

  q_lat[h]  = q_nope[h] @ W_UK[h]                    W_UK[h] is [128, 512]
  score[t]  = (q_lat[h] . c_hat[t] + q_pe[h] . kpe_hat[t]) * softmax_scale
  p[t]      = exp(score[t] - max score)
  o_lat[h]  = sum_t p[t] c_hat[t] / sum_t p[t]
  lse[h]    = max score + ln sum_t p[t]
  o[h]      = o_lat[h] @ W_UV[h]                     W_UV[h] is [512, 128]

with softmax_scale = 1/sqrt(128 + 64) by default.  The expanded path builds
K_h(t) = [c_hat[t] @ W_UK[h]^T ; kpe_hat[t]] and V_h(t) = c_hat[t] @ W_UV[h]
and runs textbook attention; it shares no arithmetic with the absorbed path
beyond the matmul primitive.  In the tutorial's notation W_i^upK (d_c x d_k)
is W_UK[h]^T and W_i^upV (d_c x d_v) is W_UV[h].

An empty context (T = 0) gives o_lat = 0, o = 0 and lse = -inf.

The prefill chunk (queries of tokens just appended, attending causally to
the positions up to their own) is the same absorbed attention per query
over its prefix; its expanded twin is the textbook masked score matrix.

Parity status: pinned (the tutorial's worked example for the row-vector
convention, absorbed == expanded, closed forms for T = 1 and for equal
scores, brute-force exp/sum on tiny inputs, split invariance; for the
prefill: absorbed == the expanded masked matrix, the first query's closed
form, causality under changes to later tokens, and a hand-computed chunk).
"""

import numpy as np

DEFAULT_SOFTMAX_SCALE = 1.0 / np.sqrt(128.0 + 64.0)


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def project_rows(x, w):
    """Row-vector convention of the tutorial: y = x @ W (x [.., k], W [k, n])."""
    return _f64(x) @ _f64(w)


def absorb_q(q_nope, w_uk):
    """q_lat[h] = q_nope[h] @ W_UK[h]; q_nope [H,128], W_UK [H,128,512]."""
    q_nope, w_uk = _f64(q_nope), _f64(w_uk)
    return np.stack([project_rows(q_nope[h], w_uk[h]) for h in range(q_nope.shape[0])])


def unabsorb_o(o_lat, w_uv):
    """o[h] = o_lat[h] @ W_UV[h]; o_lat [H,512], W_UV [H,512,128]."""
    o_lat, w_uv = _f64(o_lat), _f64(w_uv)
    return np.stack([project_rows(o_lat[h], w_uv[h]) for h in range(o_lat.shape[0])])


def scores(q_lat, q_pe, c_hat, kpe_hat, softmax_scale=DEFAULT_SOFTMAX_SCALE):
    """score[h, t] = (q_lat[h] . c_hat[t] + q_pe[h] . kpe_hat[t]) * scale."""
    return (_f64(q_lat) @ _f64(c_hat).T + _f64(q_pe) @ _f64(kpe_hat).T) * softmax_scale


def absorbed_decode(q_lat, q_pe, c_hat, kpe_hat, softmax_scale=DEFAULT_SOFTMAX_SCALE):
    """Attention of one decode query against T cached latents, all heads.

    Returns (o_lat [H, 512], lse [H]) in fp64.
    """
    q_lat = _f64(q_lat)
    H = q_lat.shape[0]
    if np.asarray(c_hat).shape[0] == 0:
        return np.zeros((H, q_lat.shape[1])), np.full(H, -np.inf)
    s = scores(q_lat, q_pe, c_hat, kpe_hat, softmax_scale)
    m = s.max(axis=1)
    p = np.exp(s - m[:, None])
    l = p.sum(axis=1)
    o_lat = (p @ _f64(c_hat)) / l[:, None]
    return o_lat, m + np.log(l)


def absorbed_decode_full(q_nope, q_pe, w_uk, w_uv, c_hat, kpe_hat,
                         softmax_scale=DEFAULT_SOFTMAX_SCALE):
    """absorb -> absorbed decode -> unabsorb.  Returns (q_lat, o_lat, lse, o)."""
    q_lat = absorb_q(q_nope, w_uk)
    o_lat, lse = absorbed_decode(q_lat, q_pe, c_hat, kpe_hat, softmax_scale)
    return q_lat, o_lat, lse, unabsorb_o(o_lat, w_uv)


def expanded_decode(q_nope, q_pe, w_uk, w_uv, c_hat, kpe_hat,
                    softmax_scale=DEFAULT_SOFTMAX_SCALE):
    """Textbook per-head attention on re-expanded K/V (tutorial "KV Cache的实现").

    Returns (o [H, 128], lse [H]).
    """
    q_nope, q_pe, w_uk, w_uv = map(_f64, (q_nope, q_pe, w_uk, w_uv))
    c_hat, kpe_hat = _f64(c_hat), _f64(kpe_hat)
    H = q_nope.shape[0]
    outs, lses = [], []
    for h in range(H):
        k_nope = c_hat @ w_uk[h].T                    # [T, 128]
        k = np.concatenate([k_nope, kpe_hat], axis=1)  # [T, 192]
        v = c_hat @ w_uv[h]                           # [T, 128]
        q = np.concatenate([q_nope[h], q_pe[h]])      # [192]
        if k.shape[0] == 0:
            outs.append(np.zeros(w_uv.shape[2]))
            lses.append(-np.inf)
            continue
        s = (k @ q) * softmax_scale
        m = s.max()
        e = np.exp(s - m)
        outs.append((e @ v) / e.sum())
        lses.append(m + np.log(e.sum()))
    return np.stack(outs), np.array(lses)


# ---------------------------------------------------------------------------
# Causal attention of a prefill chunk.
# ---------------------------------------------------------------------------

def absorbed_prefill(q_lat, q_pe, c_hat, kpe_hat, ctx_before, softmax_scale=DEFAULT_SOFTMAX_SCALE):
    """Queries of n tokens appended at positions ctx_before .. ctx_before+n-1
    of one sequence; query i attends to the cached positions 0 ..
    ctx_before + i (causal, its own token included), each one an absorbed
    decode over that prefix.  q_lat [n, H, 512], q_pe [n, H, 64]; c_hat /
    kpe_hat hold at least ctx_before + n tokens.  Returns (o_lat [n, H, 512],
    lse [n, H])."""
    n = np.asarray(q_lat).shape[0]
    outs, lses = [], []
    for i in range(n):
        t = ctx_before + i + 1
        o, l = absorbed_decode(q_lat[i], q_pe[i], c_hat[:t], kpe_hat[:t], softmax_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def expanded_prefill(q_nope, q_pe, w_uk, w_uv, c_hat, kpe_hat, ctx_before, softmax_scale=DEFAULT_SOFTMAX_SCALE):
    """Textbook masked attention of the same chunk on re-expanded K/V: per
    head, the [n, T] score matrix of [q_nope, q_pe] against [c_hat W_UK^T,
    kpe_hat], entries with key position > ctx_before + row set to -inf, a
    row softmax, times V = c_hat W_UV.  Returns (o [n, H, 128], lse [n, H])."""
    q_nope, q_pe, w_uk, w_uv = map(_f64, (q_nope, q_pe, w_uk, w_uv))
    c_hat, kpe_hat = _f64(c_hat), _f64(kpe_hat)
    n, H = q_nope.shape[0], q_nope.shape[1]
    T = ctx_before + n
    c_hat, kpe_hat = c_hat[:T], kpe_hat[:T]
    allowed = np.arange(T)[None, :] <= (ctx_before + np.arange(n))[:, None]     # [n, T]
    outs, lses = [], []
    for h in range(H):
        k = np.concatenate([c_hat @ w_uk[h].T, kpe_hat], axis=1)               # [T, 192]
        v = c_hat @ w_uv[h]                                                     # [T, 128]
        q = np.concatenate([q_nope[:, h], q_pe[:, h]], axis=1)                  # [n, 192]
        s = np.where(allowed, (q @ k.T) * softmax_scale, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        outs.append((e @ v) / e.sum(axis=1, keepdims=True))
        lses.append(m[:, 0] + np.log(e.sum(axis=1)))
    return np.stack(outs, axis=1), np.stack(lses, axis=1)


# ---------------------------------------------------------------------------
# Split-K flash-decode partials and the log-sum-exp combine.
# ---------------------------------------------------------------------------

def split_partials(q_lat, q_pe, c_hat, kpe_hat, bounds, softmax_scale=DEFAULT_SOFTMAX_SCALE):
    """Per context chunk [bounds[i], bounds[i+1]): m_i (max score), l_i
    (sum of exp(score - m_i)) and o_i (sum of exp(score - m_i) c_hat, not
    normalised).  An empty chunk has m = -inf, l = 0, o = 0."""
    q_lat = _f64(q_lat)
    H, D = q_lat.shape
    ms, ls, os_ = [], [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            ms.append(np.full(H, -np.inf)); ls.append(np.zeros(H)); os_.append(np.zeros((H, D)))
            continue
        s = scores(q_lat, q_pe, c_hat[a:b], kpe_hat[a:b], softmax_scale)
        m = s.max(axis=1)
        p = np.exp(s - m[:, None])
        ms.append(m); ls.append(p.sum(axis=1)); os_.append(p @ _f64(c_hat[a:b]))
    return np.stack(ms), np.stack(ls), np.stack(os_)


def lse_combine(m, l, o):
    """M = max_i m_i; w_i = exp(m_i - M); o_lat = sum w_i o_i / sum w_i l_i;
    lse = M + ln sum w_i l_i.  m, l: [S, H]; o: [S, H, D]."""
    m, l, o = _f64(m), _f64(l), _f64(o)
    M = m.max(axis=0)
    empty = ~np.isfinite(M)
    Ms = np.where(empty, 0.0, M)
    w = np.where(np.isfinite(m), np.exp(m - Ms[None, :]), 0.0)
    L = (w * l).sum(axis=0)
    num = (w[..., None] * o).sum(axis=0)
    o_lat = np.where(empty[:, None], 0.0, num / np.where(empty, 1.0, L)[:, None])
    lse = np.where(empty, -np.inf, Ms + np.log(np.where(empty, 1.0, L)))
    return o_lat, lse


def max_rel_error(x, ref):
    """Max over rows of ||x - ref||_inf / ||ref||_inf (rows = last axis is the
    vector).  The tolerance metric for attention outputs."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    x2 = x.reshape(-1, x.shape[-1])
    r2 = ref.reshape(-1, ref.shape[-1])
    num = np.max(np.abs(x2 - r2), axis=1)
    den = np.max(np.abs(r2), axis=1)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(num / den)) if num.size else 0.0
