"""Seeded synthetic inputs for the lightning-indexer top-k.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It holds no arithmetic of the method itself: it only draws numbers and
encodes them as the bit patterns the boundary takes (bf16 / f16 / f32, or
E4M3 codes with per-row scales), and builds the 0 / -inf additive masks the
workloads describe.

Random numbers come from SplitMix64 used as a counter-based generator
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014; constants as in Vigna's public-domain reference): value i of a
stream with seed S is mix(S + (i + 1) * 0x9E3779B97F4A7C15). Normals use the
Box-Muller transform on two consecutive uniforms. Everything is vectorised
numpy over uint64 and float64, generated in chunks so that a 1M x 128 key
cache does not need more than a few hundred MB of temporaries.

Workloads (the five shapes the indexer is exercised on; keys are already
CSA-compressed keys, queries are indexer queries):
  tiny      n_q=4 at positions 2044..2047, n_kv=2048, H=8, D=64, f16 integers
            in {-3..3}, w integers in {0..3}, causal mask, top_k=64
  decode    n_q=1, n_kv=131072, H=64, D=128, bf16 N(0,1), w ~ N(0, 1/H), mask 0
  prefill   n_q=512 at positions 15872..16383, n_kv=16384, causal
  long      n_q=2048 at positions 129024..131071, n_kv=131072, causal
  multiseq  4 rows, n_kv=1048576 shared keys, row j sees [262144 j, 262144 (j+1))
  decode_e4m3, multiseq_e4m3  the same two shapes with q and k quantised to
            E4M3 (per-row amax / 448 scales) from the same N(0, 1) draws
"""
from __future__ import annotations

import dataclasses

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

F16_ZERO = np.uint16(0x0000)
F16_NEG_INF = np.uint16(0xFC00)

# distinct stream ids per tensor of a workload
STREAM_Q, STREAM_K, STREAM_W, STREAM_SCALE = 1, 2, 3, 4

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * M1
    z = (z ^ (z >> np.uint64(27))) * M2
    return z ^ (z >> np.uint64(31))


def stream_seed(seed: int, stream: int) -> int:
    """Derive the seed of sub-stream `stream` from a workload seed."""
    with np.errstate(over="ignore"):
        z = np.array([(seed * 0x100000001B3 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return int(_mix(z + GOLDEN)[0])


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Values start .. start+count-1 of the counter-based SplitMix64 stream."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(np.uint64(seed) + i * GOLDEN)


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """Doubles in [0, 1): the top 53 bits of each SplitMix64 value."""
    return (splitmix64(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, count: int, std: float = 1.0) -> np.ndarray:
    """count N(0, std^2) doubles; element i uses stream values 2i and 2i+1 (Box-Muller)."""
    out = np.empty(count, dtype=np.float64)
    for c0 in range(0, count, _CHUNK):
        n = min(_CHUNK, count - c0)
        u = splitmix64(seed, 2 * c0, 2 * n) >> np.uint64(11)
        u1 = (u[0::2].astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
        u2 = u[1::2].astype(np.float64) * (2.0 ** -53)  # [0, 1)
        out[c0:c0 + n] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2) * std
    return out


def uniform_int(seed: int, count: int, lo: int, hi: int) -> np.ndarray:
    """count integers uniform on the inclusive set {lo, ..., hi}."""
    u = uniform01(seed, 0, count)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def f16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE binary16 bits of x (numpy's round-to-nearest-even conversion)."""
    return np.ascontiguousarray(x, dtype=np.float16).view(np.uint16)


def e4m3_values() -> np.ndarray:
    """The 127 non-negative finite E4M3 values, indexed by code 0x00..0x7E
    (OCP 8-bit floating point, E4M3 without infinities: exponent bias 7,
    exponent field 0 subnormal, 0x7F NaN); increasing with the code."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of float32 values: the nearest finite value, ties to the even
    code, magnitudes above 448 saturated to 448, the sign kept (also of 0)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    vals = e4m3_values()
    out = np.empty(x.shape, dtype=np.uint8)
    xf, of = x.reshape(-1), out.reshape(-1)
    for c0 in range(0, xf.size, _CHUNK):
        v = xf[c0:c0 + _CHUNK]
        a = np.minimum(np.abs(v.astype(np.float64)), 448.0)
        hi = np.minimum(np.searchsorted(vals, a), 126)
        lo = np.maximum(hi - 1, 0)
        d_lo, d_hi = a - vals[lo], vals[hi] - a
        code = np.where(d_hi < d_lo, hi, np.where(d_lo < d_hi, lo, np.where(hi % 2 == 0, hi, lo)))
        of[c0:c0 + v.size] = code.astype(np.uint8) | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    return out


def quantize_e4m3_rows(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-row E4M3 quantisation of float32 rows (last axis): scale = amax / 448
    in float32 (1 for an all-zero row) and codes of x / scale (float32
    division). Returns (codes uint8, same shape; scale float32, one per row)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = np.empty(x.shape, dtype=np.uint8)
    rows = x.reshape(-1, x.shape[-1])
    sc, cd = scale.reshape(-1), codes.reshape(-1, x.shape[-1])
    step = max(1, _CHUNK // max(1, x.shape[-1]))
    for r0 in range(0, rows.shape[0], step):
        cd[r0:r0 + step] = e4m3_codes(rows[r0:r0 + step] / sc[r0:r0 + step, None])
    return codes, scale


def causal_mask(n_q: int, n_kv: int, pos0: int) -> np.ndarray:
    """[n_q][n_kv] f16 bits: 0 where key s <= pos0 + t, -inf elsewhere."""
    pos = pos0 + np.arange(n_q, dtype=np.int64)[:, None]
    s = np.arange(n_kv, dtype=np.int64)[None, :]
    return np.where(s <= pos, F16_ZERO, F16_NEG_INF).astype(np.uint16)


def range_mask(n_q: int, n_kv: int, span: int) -> np.ndarray:
    """[n_q][n_kv] f16 bits: row j is 0 on [span*j, span*(j+1)) and -inf elsewhere."""
    s = np.arange(n_kv, dtype=np.int64)[None, :]
    j = np.arange(n_q, dtype=np.int64)[:, None]
    vis = (s >= span * j) & (s < span * (j + 1))
    return np.where(vis, F16_ZERO, F16_NEG_INF).astype(np.uint16)


def causal_ranges(n_q: int, pos0: int) -> tuple[np.ndarray, np.ndarray]:
    """Visible key ranges [lo, hi) per row equal to causal_mask: [0, pos0 + t + 1)."""
    lo = np.zeros(n_q, np.int32)
    hi = (pos0 + 1 + np.arange(n_q, dtype=np.int64)).astype(np.int32)
    return lo, hi


def block_ranges(n_q: int, span: int) -> tuple[np.ndarray, np.ndarray]:
    """Visible key ranges per row equal to range_mask: [span j, span (j + 1))."""
    j = np.arange(n_q, dtype=np.int64)
    return (span * j).astype(np.int32), (span * (j + 1)).astype(np.int32)


def mask_from_ranges(lo: np.ndarray, hi: np.ndarray, n_kv: int) -> np.ndarray:
    """The dense f16-bits mask of per-row ranges: 0 on [lo, hi) (clamped to
    [0, n_kv]), -inf elsewhere."""
    s = np.arange(n_kv, dtype=np.int64)[None, :]
    l = np.clip(lo.astype(np.int64), 0, n_kv)[:, None]
    h = np.clip(hi.astype(np.int64), 0, n_kv)[:, None]
    return np.where((s >= l) & (s < h), F16_ZERO, F16_NEG_INF).astype(np.uint16)


def workload_ranges(name: str):
    """The per-row ranges that stand for a workload's mask (None: no mask)."""
    if name in ("tiny", "prefill", "long"):
        n_q, n_kv = SHAPES[name][0], SHAPES[name][1]
        return causal_ranges(n_q, n_kv - n_q)
    if name in ("decode", "decode_e4m3"):
        return np.zeros(1, np.int32), np.full(1, SHAPES["decode"][1], np.int32)
    if name in ("multiseq", "multiseq_e4m3"):
        return block_ranges(4, 262144)
    raise ValueError(f"unknown workload {name!r}")


@dataclasses.dataclass
class Inputs:
    """One call's inputs as raw bit patterns (host numpy arrays).

    q_bits: [n_q, H, D] uint16 (bf16 or f16 bits, per `dtype`), or uint8
            E4M3 codes (dtype "e4m3")
    k_bits: [n_kv, D] uint16, or uint8 E4M3 codes
    w:      [n_q, H] float32
    mask:   [n_q, n_kv] uint16 f16 bits, or None (all keys visible)
    q_scale, k_scale: (dtype "e4m3" only) [n_q, H] and [n_kv] float32 row
            scales: element value = scale * code value
    """
    name: str
    dtype: str  # "bf16", "f16" or "e4m3"
    n_q: int
    n_kv: int
    H: int
    D: int
    top_k: int
    q_bits: np.ndarray
    k_bits: np.ndarray
    w: np.ndarray
    mask: np.ndarray | None
    q_scale: np.ndarray | None = None
    k_scale: np.ndarray | None = None

    @property
    def nbytes(self) -> int:
        m = 0 if self.mask is None else self.mask.nbytes
        sc = sum(a.nbytes for a in (self.q_scale, self.k_scale) if a is not None)
        return self.q_bits.nbytes + self.k_bits.nbytes + self.w.nbytes + m + sc


def _float_inputs(name, n_q, n_kv, H, D, top_k, seed, mask):
    q = f32_to_bf16_bits(normal(stream_seed(seed, STREAM_Q), n_q * H * D).astype(np.float32))
    k = f32_to_bf16_bits(normal(stream_seed(seed, STREAM_K), n_kv * D).astype(np.float32))
    w = normal(stream_seed(seed, STREAM_W), n_q * H, std=(1.0 / H) ** 0.5).astype(np.float32)
    return Inputs(name, "bf16", n_q, n_kv, H, D, top_k, q.reshape(n_q, H, D),
                  k.reshape(n_kv, D), w.reshape(n_q, H), mask)


def int_inputs(name, n_q, n_kv, H, D, top_k, seed=0, mask=None, dtype="f16",
               qk_range=(-3, 3), w_range=(0, 3)) -> Inputs:
    """Small-integer q/k (exact in f16 and bf16) and integer w."""
    qi = uniform_int(stream_seed(seed, STREAM_Q), n_q * H * D, *qk_range).astype(np.float32)
    ki = uniform_int(stream_seed(seed, STREAM_K), n_kv * D, *qk_range).astype(np.float32)
    wi = uniform_int(stream_seed(seed, STREAM_W), n_q * H, *w_range).astype(np.float32)
    enc = f16_bits if dtype == "f16" else f32_to_bf16_bits
    return Inputs(name, dtype, n_q, n_kv, H, D, top_k, enc(qi).reshape(n_q, H, D),
                  enc(ki).reshape(n_kv, D), wi.reshape(n_q, H), mask)


def float_inputs(name, n_q, n_kv, H, D, top_k, seed=0, mask=None) -> Inputs:
    """bf16 q, k ~ N(0, 1) and f32 w ~ N(0, 1/H)."""
    return _float_inputs(name, n_q, n_kv, H, D, top_k, seed, mask)


def e4m3_inputs(name, n_q, n_kv, H, D, top_k, seed=0, mask=None) -> Inputs:
    """`float_inputs`' draws (q, k ~ N(0, 1) as float32, w ~ N(0, 1/H)),
    quantised to E4M3 with one scale per q row (t, h) and per key row."""
    q = normal(stream_seed(seed, STREAM_Q), n_q * H * D).astype(np.float32).reshape(n_q, H, D)
    k = normal(stream_seed(seed, STREAM_K), n_kv * D).astype(np.float32).reshape(n_kv, D)
    w = normal(stream_seed(seed, STREAM_W), n_q * H, std=(1.0 / H) ** 0.5).astype(np.float32)
    q8, qs = quantize_e4m3_rows(q)
    del q
    k8, ks = quantize_e4m3_rows(k)
    return Inputs(name, "e4m3", n_q, n_kv, H, D, top_k, q8, k8, w.reshape(n_q, H), mask, qs, ks)


def int_e4m3_inputs(name, n_q, n_kv, H, D, top_k, seed=0, mask=None, qk_range=(-3, 3), w_range=(0, 3),
                    scale_exp=(-2, 2)) -> Inputs:
    """E4M3 codes of small integers with power-of-two row scales 2^e, e uniform
    on the inclusive `scale_exp` range, and integer w: every product and sum of
    the score is exact in float32 as well as in float64."""
    qi = uniform_int(stream_seed(seed, STREAM_Q), n_q * H * D, *qk_range).astype(np.float32)
    ki = uniform_int(stream_seed(seed, STREAM_K), n_kv * D, *qk_range).astype(np.float32)
    wi = uniform_int(stream_seed(seed, STREAM_W), n_q * H, *w_range).astype(np.float32)
    qe = uniform_int(stream_seed(seed, STREAM_SCALE), n_q * H, *scale_exp)
    ke = uniform_int(stream_seed(seed, STREAM_SCALE + 1), n_kv, *scale_exp)
    return Inputs(name, "e4m3", n_q, n_kv, H, D, top_k, e4m3_codes(qi).reshape(n_q, H, D),
                  e4m3_codes(ki).reshape(n_kv, D), wi.reshape(n_q, H), mask,
                  np.exp2(qe).astype(np.float32).reshape(n_q, H), np.exp2(ke).astype(np.float32))


def workload(name: str, seed: int = 0) -> Inputs:
    """The five named workload shapes (see the module docstring)."""
    if name == "tiny":
        return int_inputs("tiny", 4, 2048, 8, 64, 64, seed,
                          mask=causal_mask(4, 2048, 2044), dtype="f16")
    if name == "decode":
        return float_inputs("decode", 1, 131072, 64, 128, 512, seed, mask=np.zeros((1, 131072), np.uint16))
    if name == "prefill":
        return float_inputs("prefill", 512, 16384, 64, 128, 512, seed, mask=causal_mask(512, 16384, 15872))
    if name == "long":
        return float_inputs("long", 2048, 131072, 64, 128, 512, seed, mask=causal_mask(2048, 131072, 129024))
    if name == "multiseq":
        return float_inputs("multiseq", 4, 1048576, 64, 128, 512, seed, mask=range_mask(4, 1048576, 262144))
    if name == "decode_e4m3":
        return e4m3_inputs("decode_e4m3", 1, 131072, 64, 128, 512, seed, mask=np.zeros((1, 131072), np.uint16))
    if name == "multiseq_e4m3":
        return e4m3_inputs("multiseq_e4m3", 4, 1048576, 64, 128, 512, seed, mask=range_mask(4, 1048576, 262144))
    raise ValueError(f"unknown workload {name!r}")


# ------------------------------------------- the consumer: sparse attention

STREAM_QA, STREAM_KV, STREAM_SEL = 5, 6, 7


@dataclasses.dataclass
class AttnInputs:
    """Inputs of the sparse attention over the selected latent rows.

    qa_bits:   [n_q, Ha, Dc] uint16 bf16 (or f16) bits (attention queries)
    kv_bits:   [n_kv, Dc] uint16 bits of the same type (compressed latent KV rows: keys and values)
    idx:       [n_q, top_k] int32 selected rows (-1: none)
    sel_score: [n_q, top_k] float32 the selection's scores (-inf: not a selection) or None
    scale:     the softmax scale
    dtype:     "bf16" or "f16"
    """
    name: str
    n_q: int
    n_kv: int
    Ha: int
    Dc: int
    top_k: int
    qa_bits: np.ndarray
    kv_bits: np.ndarray
    idx: np.ndarray
    sel_score: np.ndarray | None
    scale: float
    dtype: str = "bf16"

    @property
    def nbytes(self) -> int:
        sc = 0 if self.sel_score is None else self.sel_score.nbytes
        return self.qa_bits.nbytes + self.kv_bits.nbytes + self.idx.nbytes + sc


def distinct_rows(seed: int, n_q: int, top_k: int, hi: np.ndarray) -> np.ndarray:
    """[n_q, top_k] int32: row t holds top_k distinct indices drawn uniformly
    from [0, hi[t]) (hi[t] >= top_k), in a random order: the positions of the
    top_k smallest of hi[t] uniform draws."""
    out = np.empty((n_q, top_k), dtype=np.int32)
    base = 0
    for t in range(n_q):
        n = int(hi[t])
        u = uniform01(seed, base, n)
        base += n
        sel = np.argpartition(u, top_k - 1)[:top_k]
        out[t] = sel[np.argsort(u[sel], kind="stable")].astype(np.int32)
    return out


def attn_inputs(name, n_q, n_kv, Ha, Dc, top_k, seed=0, pos0=None, scale=None, n_invalid=0,
                dtype="bf16") -> AttnInputs:
    """qa, kv ~ N(0, 1) in bf16 (or f16); row t selects top_k distinct keys from
    [0, pos0 + t + 1) (causal; pos0 None: from all n_kv keys); the selection
    scores are descending N(0, 1) draws; the last n_invalid selections of each
    row are turned into the two forms of "no selection" (index -1, and a valid
    index with score -inf), alternately. scale defaults to 1 / sqrt(Dc)."""
    enc = f16_bits if dtype == "f16" else f32_to_bf16_bits
    qa = enc(normal(stream_seed(seed, STREAM_QA), n_q * Ha * Dc).astype(np.float32)).reshape(n_q, Ha, Dc)
    kv = enc(normal(stream_seed(seed, STREAM_KV), n_kv * Dc).astype(np.float32)).reshape(n_kv, Dc)
    hi = np.full(n_q, n_kv, np.int64) if pos0 is None else np.minimum(pos0 + 1 + np.arange(n_q), n_kv)
    idx = distinct_rows(stream_seed(seed, STREAM_SEL), n_q, top_k, hi)
    sc = -np.sort(-normal(stream_seed(seed, STREAM_SEL + 1), n_q * top_k).reshape(n_q, top_k), axis=1)
    sc = sc.astype(np.float32)
    for j in range(top_k - n_invalid, top_k):
        if (top_k - j) % 2:
            idx[:, j] = -1
        sc[:, j] = -np.inf
    return AttnInputs(name, n_q, n_kv, Ha, Dc, top_k, qa, kv, idx, sc,
                      float(1.0 / np.sqrt(Dc)) if scale is None else float(scale), dtype)


ATTN_SHAPES = {
    # consumer of the decode and prefill selections: 64 query heads over 512-wide latent rows
    "attn_decode": (1, 131072, 64, 512, 512),
    "attn_prefill": (512, 16384, 64, 512, 512),
}


def attn_workload(name: str, seed: int = 0) -> AttnInputs:
    """The consumer's stand-in workloads: the selections of the decode and the
    prefill shapes (top-512 of their compressed keys, causal for prefill)."""
    if name == "attn_decode":
        return attn_inputs(name, 1, 131072, 64, 512, 512, seed)
    if name == "attn_prefill":
        return attn_inputs(name, 512, 16384, 64, 512, 512, seed, pos0=15872)
    raise ValueError(f"unknown workload {name!r}")


WORKLOADS = ("tiny", "decode", "prefill", "long", "multiseq")

# shape table (n_q, n_kv, H, D, top_k) without generating any data
SHAPES = {
    "tiny": (4, 2048, 8, 64, 64),
    "decode": (1, 131072, 64, 128, 512),
    "prefill": (512, 16384, 64, 128, 512),
    "long": (2048, 131072, 64, 128, 512),
    "multiseq": (4, 1048576, 64, 128, 512),
    "decode_e4m3": (1, 131072, 64, 128, 512),
    "multiseq_e4m3": (4, 1048576, 64, 128, 512),
}

# the decode and multi-sequence shapes with E4M3 q and k (one scale per row)
E4M3_WORKLOADS = ("decode_e4m3", "multiseq_e4m3")
