"""Error bounds of the tensor-core decode path, derived from its arithmetic.

The decode chunk kernel ("Strata PR #2220, attn_chunk_q8_v3_kernel": chunk
partials m, l, o of the softmax over a chunk's cells, merged by log-sum-exp)
computes, for one query row against the cells i of its (sequence, KV head):

  1. hi = f16(q), lo = f16(q - hi)         round to nearest even; the kernel's
                                            query is q' = hi + lo (|q - q'| <= 2^-22 |q|,
                                            or 2^-25 where lo is subnormal).  Windows
                                            of more than 64 rows with causal limits
                                            use q' = hi alone (u16 = 2^-11).
  2. S_i = sum_d (hi_d + lo_d) * kcode_d    products exact, summed in fp32 by
                                            the MMA (|err| <= 2 * 512 * u32 * sum(|hi| + |lo|)|k|,
                                            taken for any order and truncating adds)
  3. x_i = fma(S_i, f32(k_scale_i * scale * log2 e), 0)   two fp32 roundings
  4. p_i = ex2.approx(x_i - mref)           relative error <= 2^-20 (taken
                                            generously above the instruction's
                                            documented accuracy)
  5. P'_i = f16(p_i * v_scale_i / sigma)    relative u16 while P' is a normal
                                            f16; absolute 2^-25 when subnormal
  6. o = sigma * sum_i P'_i vcode_i, l = sum_i p_i in fp32 over a partial's
     cells (a chunk, or a run of up to RUN_CHUNKS consecutive chunks that one
     CTA accumulates), merged in fp32 with approximate exponentials (relative
     error <= 2^-20 per partial's weight).

Step 1 is removed exactly by comparing with the fp64 oracle run on the
kernel's queries q' (``refq``).  Steps 2-6 perturb cell i of a row by a
relative error eta_i of its P' and an error eps_i of its score (natural-log
units, |eps_i| <= E_i).  With softmax weights w_i and values v_id = v_scale_i *
vcode_id, to first order

  o'_d - o_d = sum_i w_i v_id eta_i + sum_i w_i (v_id - o_d) eps_i.

Bound A (any rounding):  |o'_d - o_d| <= 1.01 * (u16 * S1_d + sum_i w_i E_i (|v_id| + |o_d|)
                                              + subnormal terms) + acc_d
Bound B (every rounding error an independent mean-zero variable, the
probabilistic model of rounding-error analysis; 7 standard deviations):
  |o'_d - o_d| <= 7 * sqrt(u16^2 sum_i w_i^2 v_id^2 + sum_i w_i^2 s_i^2 (v_id - o_d)^2)
                  + subnormal terms + acc_d
where s_i bounds the standard deviation of cell i's score error: the MMA's
sum of n products has a rounding error sum_k delta_k S_k (S_k its partial
sums, |delta_k| <= u32), of standard deviation <= sqrt(n) * u32 * sum |terms|,
plus the fp32 scaling and the exponential as in E_i.
with S1_d = sum_i w_i |v_id| and acc_d = ((U + n_c) * 2 u32 + 2 * 2^-20) * (S1_d + |o_d|)
for the fp32 sums of a partial of at most U = min(RUN_CHUNKS * C, n) cells (n
the pair's cells, C the chunk size) and the merge of at most n_c = ceil(n / C)
partials (its weights in numerator and denominator), in any order.  The factor 1.01 covers
second-order terms while max E_i < 1e-2 (e^E - 1 - E <= E^2 < E / 100;
checked).

The query rounding itself (refq - ref64) has the a-priori bound
  A_q,d = 1.01 * sum_i w_i |v_id - o_d| * scale * k_scale_i * sum_d (u_q |q_d| + a_q) |kcode_d|
with u_q = 2^-22, a_q = 2^-25 for the split and u_q = u16, a_q = 2^-25 for hi alone.

P' can be subnormal only where 2^(x_i - M) * v_scale_i / max v_scale < 2^-14
(the reference mref never exceeds the row's maximum M and sigma never exceeds
the largest V scale); such a cell adds max v_scale * |vcode_id| * 2^-25 / L
(L = sum_i 2^(x_i - M) >= 1) to A, and its square to B's sum.

Everything here is test infrastructure: numpy in fp64 over the problem's
inputs.
"""
from __future__ import annotations

import numpy as np

U16 = 2.0 ** -11
U32 = 2.0 ** -24
EXP2_REL = 2.0 ** -20
LAMBDA = 7.0
SUB_MIN = 2.0 ** -14   # smallest normal f16
SUB_HALF_ULP = 2.0 ** -25
RUN_CHUNKS = 8         # chunks a CTA may accumulate into one partial


def f16_round(q: np.ndarray) -> np.ndarray:
    """Queries rounded to f16 (nearest even), as float64."""
    return np.asarray(q, np.float32).astype(np.float16).astype(np.float64)


def split_applies(p) -> bool:
    """Whether the decode kernel splits the queries into f16 hi + lo: every
    call but windows of more than 64 rows with causal limits (the rows of
    other calls go to blocks of at most 64: 16-row multiples for one
    (sequence, KV head), 24 rows for several)."""
    return getattr(p, "q_limit", None) is None or p.rows_per_kv <= 64


def kernel_queries(q: np.ndarray, split: bool) -> np.ndarray:
    """The query values the kernel multiplies, as float64: hi + lo, or hi."""
    q32 = np.asarray(q, np.float32)
    hi = q32.astype(np.float16).astype(np.float32)
    if not split:
        return hi.astype(np.float64)
    lo = (q32 - hi).astype(np.float16).astype(np.float64)  # q - hi is exact in fp32
    return hi.astype(np.float64) + lo


def cells_of(p, b: int, g: int):
    """Codes and scales of the valid cells of (sequence b, KV head g), in list order."""
    sel = p.sel_of(b).astype(np.int64)
    P = int(getattr(p, "page_cells", 1))
    ok = (sel >= 0) & (sel < p.page_table_len * P)
    pos = sel[ok]
    ent = p.page_table[b][pos // P].astype(np.int64)
    ok2 = (ent >= 0) & (ent < p.pool_cells // P)
    slot = ent[ok2] * P + pos[ok2] % P
    kc = p.k_pool[b, g, slot].astype(np.float64)
    vc = p.v_pool[b, g, slot].astype(np.float64)
    ks = p.k_scale[b, g, slot].astype(np.float64)
    vs = p.v_scale[b, g, slot].astype(np.float64)
    return kc, vc, ks, vs


def bounds(p, q_rows: np.ndarray, b: int, g: int, split: bool = True, run_chunks: int = RUN_CHUNKS):
    """Bounds A, B (steps 2-6) and A_q (step 1) for the query rows q_rows
    [R][D] (fp32 values) of (sequence b, KV head g): arrays [R][D], plus the
    largest E_i.  run_chunks: chunks that one partial may span."""
    kc, vc, ks, vs = cells_of(p, b, g)
    R, D = q_rows.shape
    if kc.shape[0] == 0:
        z = np.zeros((R, D))
        return z, z, z, 0.0
    q64 = np.asarray(q_rows, np.float64)
    q16 = kernel_queries(q_rows, split)
    scale = float(p.softmax_scale)
    x = scale * (q16 @ kc.T) * ks[None, :]               # natural-log units, [R][n]
    M = x.max(axis=1, keepdims=True)
    e = np.exp(x - M)
    L = e.sum(axis=1, keepdims=True)
    w = e / L
    v = vc * vs[:, None]                                  # [n][D]
    av = np.abs(v)
    o = w @ v
    S1 = w @ av
    # score error per (row, cell): MMA sum, the two fp32 roundings, the exponential
    nsum = 512 if split else 256  # products the MMA sums per score
    hi = kernel_queries(q_rows, False)
    mag = np.abs(hi) + np.abs(q16 - hi)  # |hi| + |lo| (lo = 0 for hi alone)
    E = (scale * ks[None, :] * 2 * nsum * U32 * (mag @ np.abs(kc).T)
         + 2 * U32 * np.abs(x) + EXP2_REL)
    WE = w * E
    # subnormal P': possible only where this lower bound of P' is below 2^-14
    vmax = float(np.abs(vs).max())
    flag = (e * np.abs(vs)[None, :] / vmax) < SUB_MIN
    a_scale = vmax * SUB_HALF_ULP
    A_sub = a_scale * ((flag / L) @ np.abs(vc))
    B_sub = a_scale * np.sqrt((flag / L ** 2) @ (vc * vc))
    C = int(p.chunk_cells)
    n = kc.shape[0]
    U = min(run_chunks * C, n)
    acc = ((U + -(-n // C)) * 2 * U32 + 2 * EXP2_REL) * (S1 + np.abs(o))
    A = 1.01 * (U16 * S1 + WE @ av + np.abs(o) * WE.sum(axis=1, keepdims=True) + A_sub) + acc
    sd = (scale * ks[None, :] * np.sqrt(nsum) * U32 * (mag @ np.abs(kc).T)
          + 2 * U32 * np.abs(x) + EXP2_REL)
    WS2 = (w * sd) ** 2
    cterm = (WS2 @ (v * v)) - 2 * o * (WS2 @ v) + o * o * WS2.sum(axis=1, keepdims=True)
    B = LAMBDA * np.sqrt(U16 * U16 * ((w * w) @ (v * v)) + np.maximum(cterm, 0.0)) + LAMBDA * B_sub + acc
    # step 1, a priori: |x' - x| <= scale * ks * sum (u_q |q| + a_q) |k|
    u_q = 2.0 ** -22 if split else U16
    Eq = scale * ks[None, :] * ((u_q * np.abs(q64) + SUB_HALF_ULP) @ np.abs(kc).T)
    Aq = 1.01 * ((w * Eq) @ av + np.abs(o) * (w * Eq).sum(axis=1, keepdims=True))
    return A, B, Aq, float(E.max())


def problem_bounds(p, split: bool = None, run_chunks: int = RUN_CHUNKS):
    """Bounds for every output row of a decode problem (f32 queries, no causal
    limits): A, B, A_q shaped like the output [B][T][G*H][D], and max E.
    ``split``: the kernel's query split (default: as the kernel takes it);
    ``run_chunks``: chunks that one partial may span (1: a partial per chunk)."""
    if split is None:
        split = split_applies(p)
    T, G, H, D = p.n_queries, p.n_kv_heads, p.q_per_kv, p.head_dim
    shp = (p.n_seq, T, G * H, D)
    A, B, Aq = np.zeros(shp), np.zeros(shp), np.zeros(shp)
    emax = 0.0
    q = np.asarray(p.q, np.float32)
    for b in range(p.n_seq):
        for g in range(G):
            rows = q[b, :, g * H:(g + 1) * H, :].reshape(T * H, D)
            a, bb, aq, em = bounds(p, rows, b, g, split, run_chunks)
            A[b, :, g * H:(g + 1) * H, :] = a.reshape(T, H, D)
            B[b, :, g * H:(g + 1) * H, :] = bb.reshape(T, H, D)
            Aq[b, :, g * H:(g + 1) * H, :] = aq.reshape(T, H, D)
            emax = max(emax, em)
    return A, B, Aq, emax


def with_kernel_queries(p, split: bool = None):
    """A copy of problem p whose fp32 queries are the values the kernel
    multiplies (hi + lo, exact in fp32, or hi)."""
    import copy
    if split is None:
        split = split_applies(p)
    pq = copy.copy(p)
    pq.q = kernel_queries(p.q, split).astype(np.float32)
    return pq


def row_norm_errors(out, ref):
    """Per output row ||out - ref|| / ||ref|| (rows of D values)."""
    out = np.asarray(out, np.float64).reshape(-1, np.shape(out)[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, np.shape(ref)[-1])
    return np.linalg.norm(out - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-300)


def split_visible(out, ref_split, ref_hi) -> bool:
    """Whether an output follows the queries' hi + lo (True) or hi alone
    (False): the mean absolute error against the oracle on each, compared."""
    out = np.asarray(out, np.float64)
    a = float(np.mean(np.abs(out - np.asarray(ref_split))))
    b = float(np.mean(np.abs(out - np.asarray(ref_hi))))
    return a < b
