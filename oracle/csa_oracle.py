"""fp64 CPU oracle for the CSA / HCA hybrid compressed attention.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU-baseline / reference legs
of bench.py may import this module. The CUDA library never calls it and shares no code with it.

What it computes, and where the pages state it:
  * CSA: every m=4 consecutive KV tokens are merged into one compressed entry; a Lightning
    Indexer scores the entries, a per-query top-k keeps some of them, and attention runs over the
    kept entries plus a sliding window of n_win=128 raw tokens.
      - Lighthouse, "deep deepseek v4 release", section 八.3 (CSA with m=4, top-k 1024/512,
        sliding-window branch n_win=128)
      - 9fzt.com DeepSeek-V4 summary, item 1) (CSA: compress along the sequence, then sparse
        selection) and item 4) (FP4 indexer QK path, index scores reduced from FP32 to BF16)
      - blog.tulong.co DeepSeek-V4 Q&A, "技术架构创新" 1 (4 tokens per block)
  * HCA: every m'=128 tokens form one entry; attention is dense over all entries plus the window.
      - Lighthouse section 八.3 (m'=128, dense, no top-k); blog.tulong.co "技术架构创新" 1.
  * The two layer types alternate along depth (Lighthouse 八.3; elebank "DeepSeek-V4 explained",
    模型創新 1).

Where the pages are silent, this file takes the readings below (each is listed with its reason in
the design notes of the repository):
  R1 blocks are aligned and non-overlapping, [j*m, (j+1)*m); E = floor(N/m); a partial trailing
     block is not an entry.
  R2 pooling = softmax over the block's m per-token scalar logits; the same weights pool K and V.
  R3 a query at position t sees entry j iff (j+1)*m - 1 <= t.
  R4 window(t) = raw tokens [max(0, t-W+1), t].
  R5 entries and window tokens form one softmax over their multiset (no de-duplication).
  R6 index score s[t,j] = sum_h ReLU(q_I[t,h] . k_I[j]) with FP4 (e2m1) values times UE8M0
     per-32 scales; exact in FP32, then rounded to BF16 with round-to-nearest-even.
  R7 top-k order: (score descending, index ascending); take min(k, visible); output sorted
     ascending, padded with -1.
  R8 logits are q.k with no extra scale (1/sqrt(d) is folded into Q).
  R9 an empty attention set (W = 0 and no visible entry) gives output 0 and LSE = -inf.
  R14 the indexer's own keys are pooled from per-token index-key rows with the KV entries'
     block pooling (R2), rounded to bf16, and converted to MX FP4 with the OCP MX v1.0 rule
     (block scale 2^(floor(log2 amax) - 2), elements rounded to nearest-even on the e2m1 grid,
     saturating at 6).

Parity unpinned (readings with nothing on the pages to check them against; the arithmetic that
implements them is pinned by the tests): the R6 score formula itself (which nonlinearity, unit
head weights) and R14's use of the layer's pooling logits for the index keys.

Everything is plain numpy in float64; bf16 tensors arrive as uint16 bit arrays.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Tuple

import numpy as np

# e2m1 (FP4) magnitudes for the 3 low bits of a code; bit 3 is the sign. The encoding is the
# OCP Microscaling Formats (MX) v1.0 FP4 E2M1 element format: 2 exponent bits with bias 1,
# 1 mantissa bit, exponent 0 holding the subnormal 0.5 * mantissa.
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
MX_BLOCK = 32          # one UE8M0 scale per 32 consecutive elements (OCP MX block size)


# ----------------------------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64. A bf16 value is the upper half of an fp32."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_rne(x) -> np.ndarray:
    """Round float64 values that are exactly representable in fp32 to bf16 bits with
    round-to-nearest, ties-to-even (the rounding the index-score path applies, 9fzt.com item 4).
    -0 is returned as +0. Values must be finite."""
    x = np.asarray(x, dtype=np.float64) + 0.0          # -0 -> +0
    f = x.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), x):
        raise ValueError("value not exactly representable in fp32")
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def e2m1_unpack(codes, n: int) -> np.ndarray:
    """Packed FP4 codes [..., n/2] uint8 -> values [..., n] float64. The low nibble of byte i is
    element 2i, the high nibble element 2i+1."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] * 2 == n
    lo = codes & np.uint8(0x0F)
    hi = codes >> np.uint8(4)
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (n,))
    sign = np.where(nib & np.uint8(0x8), -1.0, 1.0)
    return sign * E2M1_MAGNITUDES[nib & np.uint8(0x7)]


def ue8m0_to_f64(scales) -> np.ndarray:
    """UE8M0 scale bytes -> 2^(s-127). 255 (NaN in the MX format) is rejected."""
    s = np.asarray(scales, dtype=np.int64)
    if np.any(s == 255):
        raise ValueError("UE8M0 NaN scale")
    return np.ldexp(1.0, s - 127)


def mx_fp4_dequant(codes, scales, n: int) -> np.ndarray:
    """Block-scaled FP4 vectors: value[i] = e2m1(code[i]) * 2^(scale[i // 32] - 127)."""
    v = e2m1_unpack(codes, n)
    sc = np.repeat(ue8m0_to_f64(scales), MX_BLOCK, axis=-1)
    assert sc.shape == v.shape
    return v * sc


def f64_to_bf16_rne_any(x) -> np.ndarray:
    """Round arbitrary finite float64 values straight to bf16 bits (8 significant bits) with
    round-to-nearest, ties-to-even; one rounding, no detour through fp32. Values must be 0 or
    at least 2^-126 in magnitude (no bf16 subnormals) and below the bf16 maximum."""
    x = np.asarray(x, dtype=np.float64)
    f, k = np.frexp(x)                      # x = f * 2^k, 0.5 <= |f| < 1
    if np.any((x != 0) & (np.abs(x) < 2.0 ** -126)):
        raise ValueError("bf16 subnormal result")
    r = np.ldexp(np.rint(np.ldexp(f, 8)), k - 8)  # np.rint rounds half to even
    r = r + 0.0                              # -0 -> +0
    f32 = r.astype(np.float32)
    if not np.all(np.isfinite(f32)):
        raise ValueError("bf16 overflow")
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# MX FP4 conversion (OCP Microscaling Formats v1.0, section 6.3, "conversion to MX": the shared
# scale of a 32-element block is X = 2^(floor(log2(max_i |V_i|)) - emax_elem), with emax_elem = 2
# for FP4 E2M1 (largest normal 6 = 1.5 * 2^2); each element is V_i / X rounded to the element
# format with round-to-nearest-even, magnitudes above the largest normal clamped to it).
E2M1_EMAX = 2


def e2m1_round(y) -> np.ndarray:
    """float64 -> 4-bit e2m1 codes: the nearest of the 8 magnitudes, a tie going to the even
    code (mantissa bit 0), magnitudes beyond 6 saturating to 6; the sign bit copies the sign of
    the input (a negative value that rounds to zero gives code 8, -0)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), E2M1_MAGNITUDES[-1])
    dist = np.abs(a[..., None] - E2M1_MAGNITUDES)          # [..., 8]
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best                                     # one or two nearest magnitudes
    even = cand & (np.arange(8) % 2 == 0)
    idx = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    sign = np.signbit(y).astype(np.int64)
    return (idx + 8 * sign).astype(np.uint8)


def mx_fp4_quantize(x) -> Tuple[np.ndarray, np.ndarray]:
    """x [..., n] float64, n % 32 == 0 -> (packed e2m1 codes [..., n/2] uint8, UE8M0 scale bytes
    [..., n/32] uint8); MX FP4 conversion as stated above. An all-zero block gets the smallest
    scale (byte 0, 2^-127) and zero codes; the exponent is clamped to the UE8M0 range
    [-127, 127]."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    assert n % MX_BLOCK == 0
    blk = x.reshape(x.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    amax = np.abs(blk).max(axis=-1)
    _, k = np.frexp(amax)                                   # amax = f * 2^k, f in [0.5, 1)
    e = np.where(amax > 0, (k - 1) - E2M1_EMAX, -127)       # floor(log2(amax)) - emax_elem
    e = np.clip(e, -127, 127)
    y = blk / np.ldexp(1.0, e)[..., None]
    codes = e2m1_round(y).reshape(x.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << np.uint8(4))).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


# ----------------------------------------------------------------------------------------------
# compression (CSA m=4, HCA m=128)
# ----------------------------------------------------------------------------------------------
def entry_count(N: int, m: int) -> int:
    """R1: number of complete, aligned blocks of m tokens in N tokens."""
    return N // m


def pooling_weights(logits_block: np.ndarray) -> np.ndarray:
    """R2: softmax over the m per-token logits of one block (last axis)."""
    w = np.asarray(logits_block, dtype=np.float64)
    e = np.exp(w - w.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def compress(raw: np.ndarray, logits: np.ndarray, m: int) -> np.ndarray:
    """Pool one sequence's raw rows [N, d] into entries [E, d]:
    entry[j] = sum_i softmax(w[jm .. jm+m-1])_i * raw[jm+i]   (Lighthouse 八.3; R1, R2)."""
    raw = np.asarray(raw, dtype=np.float64)
    N, d = raw.shape
    E = entry_count(N, m)
    p = pooling_weights(np.asarray(logits, dtype=np.float64)[: E * m].reshape(E, m))
    return np.einsum("ji,jid->jd", p, raw[: E * m].reshape(E, m, d))


def index_key_entries(xi_bits, logits, m: int):
    """The Lightning Indexer's own compressed keys (Lighthouse 八.7 lists them beside the CSA and
    HCA entries; 9fzt.com item 4 puts the indexer's QK path in FP4): one sequence's raw index-key
    rows [N, d_I] (bf16 bits) are pooled with the block-pooling operator of the KV entries (R2,
    the same per-token logits), each pooled value is rounded to bf16, and every entry is
    converted to MX FP4 (R14). Returns (codes [E, d_I/2], scales [E, d_I/32], pooled bf16 bits
    [E, d_I], pooled float64 [E, d_I])."""
    pooled = compress(bf16_to_f64(xi_bits), logits, m)
    pb = f64_to_bf16_rne_any(pooled)
    codes, scales = mx_fp4_quantize(bf16_to_f64(pb))
    return codes, scales, pb, pooled


# ----------------------------------------------------------------------------------------------
# Lightning Indexer scores and top-k
# ----------------------------------------------------------------------------------------------
def visible_entries(t: int, m: int, E: int) -> int:
    """R3: entries j with (j+1)*m - 1 <= t, capped by the E entries that exist."""
    return max(0, min(E, (t + 1) // m))


def index_scores(qi_codes, qi_scales, ki_codes, ki_scales, d_I: int) -> np.ndarray:
    """One query's scores over entries: s[j] = sum_h max(q_h . k_j, 0)  (R6).
    qi_codes [H_I, d_I/2], qi_scales [H_I, d_I/32]; ki_codes [E, d_I/2], ki_scales [E, d_I/32].
    Returns float64 values, each checked to be exactly representable in fp32."""
    q = mx_fp4_dequant(qi_codes, qi_scales, d_I)          # [H_I, d_I]
    k = mx_fp4_dequant(ki_codes, ki_scales, d_I)          # [E, d_I]
    dots = k @ q.T                                        # [E, H_I]
    s = np.maximum(dots, 0.0).sum(axis=1) + 0.0
    if not np.array_equal(s.astype(np.float32).astype(np.float64), s):
        raise AssertionError("index score not exact in fp32")
    return s


def topk_select(score_bits, n_visible: int, k: int) -> Tuple[np.ndarray, int]:
    """R7: the min(k, n_visible) entries with the largest BF16 score, ties to the lower index,
    returned sorted ascending and padded with -1 to length k."""
    return topk_select_values(bf16_to_f64(np.asarray(score_bits)[:n_visible]), n_visible, k)


def topk_select_values(values, n_visible: int, k: int) -> Tuple[np.ndarray, int]:
    """R7 on real-valued scores (the FP32 scores the pages' BF16 rounding replaces, 9fzt.com
    item 4): the min(k, n_visible) largest, ties (-0 equal to +0) to the lower index, sorted
    ascending and padded with -1."""
    vals = np.asarray(values, dtype=np.float64)[:n_visible] + 0.0
    order = np.lexsort((np.arange(n_visible), -vals))     # primary: -score, secondary: index
    cnt = min(k, n_visible)
    idx = np.full(k, -1, dtype=np.int64)
    idx[:cnt] = np.sort(order[:cnt])
    return idx, cnt


# ----------------------------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------------------------
def window_tokens(t: int, W: int) -> np.ndarray:
    """R4: raw positions max(0, t-W+1) .. t."""
    return np.arange(max(0, t - W + 1), t + 1, dtype=np.int64)


def attention_weights(q: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """softmax over the key set of q.k (R8): q [H, d], keys [n, d] -> [H, n]."""
    logits = q @ keys.T
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """out[h] = sum_n softmax_n(q_h . key_n) value_n and lse[h] = log sum_n exp(q_h . key_n).
    An empty key set gives zeros and -inf (R9)."""
    q = np.asarray(q, dtype=np.float64)
    H, d = q.shape
    if keys.shape[0] == 0:
        return np.zeros((H, values.shape[1])), np.full(H, -np.inf)
    logits = q @ keys.T
    mx = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - mx)
    z = e.sum(axis=1, keepdims=True)
    return (e / z) @ values, (mx + np.log(z))[:, 0]


def csa_attend_one(q, k_cmp, v_cmp, idx, cnt, k_raw, v_raw, t, W):
    """CSA attention of one query at position t (Lighthouse 八.3; R4, R5):
    keys = {k_cmp[j] : j in idx[:cnt]} + {k_raw[u] : u in window(t)}."""
    sel = np.asarray(idx[:cnt], dtype=np.int64)
    win = window_tokens(t, W)
    keys = np.concatenate([k_cmp[sel], k_raw[win]], axis=0)
    vals = np.concatenate([v_cmp[sel], v_raw[win]], axis=0)
    return attend(q, keys, vals)


def hca_attend_one(q, k_cmp, v_cmp, n_vis, k_raw, v_raw, t, W):
    """HCA attention of one query at position t (Lighthouse 八.3: dense over all visible
    entries, no top-k; R4, R5)."""
    win = window_tokens(t, W)
    keys = np.concatenate([k_cmp[:n_vis], k_raw[win]], axis=0)
    vals = np.concatenate([v_cmp[:n_vis], v_raw[win]], axis=0)
    return attend(q, keys, vals)


# ----------------------------------------------------------------------------------------------
# whole layers (one sequence at a time; arrays are numpy, bf16 as uint16 bits)
# ----------------------------------------------------------------------------------------------
def csa_layer_seq(q_bits, k_raw_bits, v_raw_bits, logits, qi_codes, qi_scales, ki_codes,
                  ki_scales, *, m, W, k, d_I, q_pos0, query_rows=None,
                  k_cmp=None, v_cmp=None) -> Dict[str, np.ndarray]:
    """CSA layer for one sequence.

    q_bits [Nq, H, d]; k_raw_bits, v_raw_bits [N, d]; logits [N]; qi_* [Nq, H_I, ...];
    ki_* [E, ...]. Entries are pooled here in float64 unless k_cmp / v_cmp are given (e.g. the
    bf16 entries another implementation stored, as float64). `query_rows` restricts the work to
    a subset of the Nq queries. Returns per computed query: out [n, H, d], lse [n, H],
    scores (bf16 bits, visible part only, list), idx [n, k], cnt [n]."""
    k_raw = bf16_to_f64(k_raw_bits)
    v_raw = bf16_to_f64(v_raw_bits)
    N = k_raw.shape[0]
    E = entry_count(N, m)
    if k_cmp is None:
        k_cmp = compress(k_raw, logits, m)
    if v_cmp is None:
        v_cmp = compress(v_raw, logits, m)
    Nq = q_bits.shape[0]
    rows = range(Nq) if query_rows is None else query_rows
    outs, lses, idxs, cnts, scores = [], [], [], [], []
    for i in rows:
        t = q_pos0 + i
        n_vis = visible_entries(t, m, E)
        s = index_scores(qi_codes[i], qi_scales[i], ki_codes[:n_vis], ki_scales[:n_vis], d_I)
        sb = f64_to_bf16_rne(s)
        idx, cnt = topk_select(sb, n_vis, k)
        o, l = csa_attend_one(bf16_to_f64(q_bits[i]), k_cmp, v_cmp, idx, cnt, k_raw, v_raw, t, W)
        outs.append(o); lses.append(l); idxs.append(idx); cnts.append(cnt); scores.append(sb)
    return {"out": np.stack(outs), "lse": np.stack(lses), "idx": np.stack(idxs),
            "cnt": np.array(cnts), "scores": scores}


def hca_layer_seq(q_bits, k_raw_bits, v_raw_bits, logits, *, m, W, q_pos0, query_rows=None,
                  k_cmp=None, v_cmp=None) -> Dict[str, np.ndarray]:
    """HCA layer for one sequence (same conventions as csa_layer_seq)."""
    k_raw = bf16_to_f64(k_raw_bits)
    v_raw = bf16_to_f64(v_raw_bits)
    N = k_raw.shape[0]
    E = entry_count(N, m)
    if k_cmp is None:
        k_cmp = compress(k_raw, logits, m)
    if v_cmp is None:
        v_cmp = compress(v_raw, logits, m)
    Nq = q_bits.shape[0]
    rows = range(Nq) if query_rows is None else query_rows
    outs, lses = [], []
    for i in rows:
        t = q_pos0 + i
        o, l = hca_attend_one(bf16_to_f64(q_bits[i]), k_cmp, v_cmp, visible_entries(t, m, E),
                              k_raw, v_raw, t, W)
        outs.append(o); lses.append(l)
    return {"out": np.stack(outs), "lse": np.stack(lses)}
