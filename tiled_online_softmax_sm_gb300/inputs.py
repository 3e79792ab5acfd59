"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it draws random numbers, rounds
them to the storage type, and lays them out.  Both the CUDA path and the CPU
oracle receive the arrays it produces, so neither side generates its own data.

Random numbers: numpy's Philox-4x32-10 bit generator, keyed by a SeedSequence
of (seed, stream, tensor) so that every tensor of every workload has its own
reproducible stream.  Normals come from numpy's ``standard_normal`` (float32).

bf16 storage: float32 -> bf16 with round-to-nearest-even on the bit pattern;
the oracle receives the exact float32 widening of those bf16 values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BASE_SEED = 42  # the worked example of "FlashAttention推理优化实战100例 01" seeds with 42


def rng(seed: int, stream: int = 0, tensor: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream, tensor])))


def normal_f32(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(size=shape, dtype=np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    bits = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        bits[nan] = np.uint16(0x7FC0)
    return bits


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 value (kept in float32)."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


def _e4m3_table():
    """The 254 finite e4m3 (FP8, 4 exponent bits, bias 7, 3 mantissa bits) values
    by code, NaN (0x7f, 0xff) excluded: code -> value."""
    codes = np.arange(256, dtype=np.int64)
    s = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = codes & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7)) * s
    finite = (codes & 0x7F) != 0x7F
    return codes[finite], val[finite]


_E4M3_CODES, _E4M3_VALUES = _e4m3_table()
E4M3_MAX = 448.0


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to the even code), saturating at
    +-448 (the satfinite convention); returns uint8 codes."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    pos = _E4M3_VALUES >= 0
    pc, pv = _E4M3_CODES[pos], _E4M3_VALUES[pos]
    order = np.argsort(pv, kind="stable")
    pc, pv = pc[order], pv[order]
    # +0 and -0 both appear; keep +0 (code 0) for the magnitude lookup
    keep = np.concatenate([[True], np.diff(pv) > 0])
    pc, pv = pc[keep], pv[keep]
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(pv, a), 1, len(pv) - 1)
    lo = hi - 1
    dlo, dhi = a - pv[lo], pv[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((pc[hi] & 1) == 0))
    code = np.where(pick_hi, pc[hi], pc[lo]).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return code


def e4m3_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    lut = np.zeros(256, np.float32)
    lut[_E4M3_CODES] = _E4M3_VALUES.astype(np.float32)
    lut[0x7F] = lut[0xFF] = np.nan
    return lut[np.asarray(bits, dtype=np.uint8)]


@dataclass
class Tensor:
    """One input tensor: storage bits (bf16 as uint16, or float32) plus the
    exact float32 values the oracle reads."""
    dtype: str            # "bf16", "f32" or "e4m3"
    data: np.ndarray      # uint16 for bf16, float32 for f32, uint8 codes for e4m3
    values: np.ndarray    # float32, exact (for e4m3: code value * descale)
    descale: float = 1.0  # e4m3: stored value * descale = value

    @staticmethod
    def from_f32(x: np.ndarray, dtype: str) -> "Tensor":
        if dtype == "bf16":
            bits = f32_to_bf16_bits(x)
            return Tensor("bf16", bits, bf16_bits_to_f32(bits))
        if dtype == "f32":
            x = np.ascontiguousarray(x, dtype=np.float32)
            return Tensor("f32", x, x)
        if dtype == "e4m3":
            # per-tensor amax scaling by a power of two (so code * descale is
            # exact in fp32): the largest magnitude lands in (224, 448]
            amax = float(np.max(np.abs(x))) if x.size else 0.0
            descale = float(2.0 ** np.ceil(np.log2(amax / E4M3_MAX))) if amax > 0 else 1.0
            codes = f32_to_e4m3_bits(np.asarray(x, np.float64) / descale)
            vals = (e4m3_bits_to_f32(codes).astype(np.float64) * descale).astype(np.float32)
            return Tensor("e4m3", codes, vals, descale)
        raise ValueError(dtype)


@dataclass
class DenseCase:
    q: Tensor
    k: Tensor
    v: Tensor
    B: int
    H: int
    Hkv: int
    n: int
    m: int
    d: int
    dv: int
    scale: float          # float32 value, as passed to the library
    causal: bool
    name: str = ""


def fp32_scale(d: int) -> float:
    """1/sqrt(d) rounded to float32: the value the library receives.

    The oracle widens this same float32 value, so both sides use one scale
    (the float64-promotion trap of "手搓 Attention" §4)."""
    return float(np.float32(1.0 / math.sqrt(d)))


def dense_case(seed: int, B: int, H: int, n: int, m: int, d: int, dv: int | None = None,
               Hkv: int | None = None, dtype: str = "bf16", causal: bool = False,
               hot: float = 1.0, stream: int = 0, scale: float | None = None,
               name: str = "") -> DenseCase:
    """Q [B,n,H,d], K [B,m,Hkv,d], V [B,m,Hkv,dv], iid N(0,1); Q and K are
    multiplied by ``hot`` before rounding (the x10 'hot' inputs)."""
    dv = d if dv is None else dv
    Hkv = H if Hkv is None else Hkv
    q = normal_f32(rng(seed, stream, 0), (B, n, H, d))
    k = normal_f32(rng(seed, stream, 1), (B, m, Hkv, d))
    v = normal_f32(rng(seed, stream, 2), (B, m, Hkv, dv))
    if hot != 1.0:
        q *= np.float32(hot)
        k *= np.float32(hot)
    return DenseCase(Tensor.from_f32(q, dtype), Tensor.from_f32(k, dtype), Tensor.from_f32(v, dtype),
                     B, H, Hkv, n, m, d, dv, fp32_scale(d) if scale is None else scale, causal, name)


@dataclass
class VarlenCase:
    q: Tensor
    k: Tensor
    v: Tensor
    cu_seqlens: np.ndarray  # int32 [S+1], shared by Q and K (self-attention prefill)
    lens: np.ndarray
    H: int
    Hkv: int
    d: int
    dv: int
    scale: float
    causal: bool
    hot_rows_q: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))
    hot_rows_k: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))


def varlen_case(seed: int, lens, H: int, d: int, dv: int | None = None, Hkv: int | None = None,
                hot_frac: float = 0.10, hot: float = 20.0, causal: bool = True,
                stream: int = 5) -> VarlenCase:
    """Packed [total,H,d] self-attention inputs; independently for Q and K a
    seeded ``hot_frac`` of token rows (all heads of the token) is multiplied
    by ``hot`` before rounding to bf16.  V is not scaled."""
    dv = d if dv is None else dv
    Hkv = H if Hkv is None else Hkv
    lens = np.asarray(lens, dtype=np.int64)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    q = normal_f32(rng(seed, stream, 0), (T, H, d))
    k = normal_f32(rng(seed, stream, 1), (T, Hkv, d))
    v = normal_f32(rng(seed, stream, 2), (T, Hkv, dv))
    n_hot = int(round(hot_frac * T))
    hq = np.sort(rng(seed, stream, 3).choice(T, size=n_hot, replace=False)) if T else np.zeros(0, np.int64)
    hk = np.sort(rng(seed, stream, 4).choice(T, size=n_hot, replace=False)) if T else np.zeros(0, np.int64)
    q[hq] *= np.float32(hot)
    k[hk] *= np.float32(hot)
    return VarlenCase(Tensor.from_f32(q, "bf16"), Tensor.from_f32(k, "bf16"), Tensor.from_f32(v, "bf16"),
                      cu, lens, H, Hkv, d, dv, fp32_scale(d), causal, hq, hk)


def uniform_lengths(seed: int, count: int, lo: int, hi: int, stream: int = 0, tensor: int = 9):
    """count integers uniform on [lo, hi] inclusive."""
    return rng(seed, stream, tensor).integers(lo, hi + 1, size=count).astype(np.int64)


@dataclass
class DecodeCase:
    q: Tensor                 # [S,H,d]
    k_cache: Tensor           # [P,Hkv,page,d]
    v_cache: Tensor           # [P,Hkv,page,dv]
    block_table: np.ndarray   # int32 [S,max_blocks]; -1 past each sequence's pages
    seq_lens: np.ndarray      # int32 [S]
    H: int
    Hkv: int
    d: int
    dv: int
    page_size: int
    num_pages: int
    max_blocks: int
    scale: float

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V for every valid token (the algorithmic KV traffic)."""
        return int(self.seq_lens.sum()) * self.Hkv * (self.d + self.dv) * 2


def decode_case(seed: int, num_seqs: int, H: int, Hkv: int, d: int, dv: int | None = None,
                page_size: int = 16, len_lo: int = 512, len_hi: int = 8192,
                lens=None, unused_frac: float = 0.10, max_blocks: int | None = None,
                poison: bool = True, stream: int = 3) -> DecodeCase:
    """Paged KV cache with a shared page pool.

    Context lengths are uniform on [len_lo, len_hi] (or given).  The pool holds
    the pages every sequence uses plus ``unused_frac`` more; a random
    permutation of the pool's ids is cut into consecutive slices, one per
    sequence, so each block table is a random set of physical pages in random
    order.  K/V values are iid N(0,1) rounded to bf16.  With ``poison``, the
    unused pages and the slots past each sequence's end in its last page hold
    NaN, so any stray read shows up as NaN in the output.
    """
    dv = d if dv is None else dv
    if lens is None:
        lens = uniform_lengths(seed, num_seqs, len_lo, len_hi, stream, 9)
    lens = np.asarray(lens, dtype=np.int64)
    pages_per = (lens + page_size - 1) // page_size
    used = int(pages_per.sum())
    P = used + int(math.ceil(unused_frac * used))
    P = max(P, 1)
    if max_blocks is None:
        max_blocks = max(1, int(pages_per.max()) if len(pages_per) else 1)
    perm = rng(seed, stream, 10).permutation(P).astype(np.int32)
    table = np.full((len(lens), max_blocks), -1, np.int32)
    off = 0
    for s, np_ in enumerate(pages_per):
        table[s, :np_] = perm[off:off + np_]
        off += int(np_)
    q = normal_f32(rng(seed, stream, 0), (len(lens), H, d))
    kc = normal_f32(rng(seed, stream, 1), (P, Hkv, page_size, d))
    vc = normal_f32(rng(seed, stream, 2), (P, Hkv, page_size, dv))
    if poison:
        unused = perm[used:]
        kc[unused] = np.nan
        vc[unused] = np.nan
        for s, L in enumerate(lens):
            tail = int(L % page_size)
            if tail and pages_per[s] > 0:
                last = table[s, pages_per[s] - 1]
                kc[last, :, tail:, :] = np.nan
                vc[last, :, tail:, :] = np.nan
    return DecodeCase(Tensor.from_f32(q, "bf16"), Tensor.from_f32(kc, "bf16"), Tensor.from_f32(vc, "bf16"),
                      table, lens.astype(np.int32), H, Hkv, d, dv, page_size, P, max_blocks,
                      fp32_scale(d))


# Named workloads (sizes from the pages' configurations).
def c1_fp32(hot: bool = False, seed: int = BASE_SEED) -> DenseCase:
    """Single-head non-causal fp32: n=m=256, d=dv=64, scale 1/8 (+ x10 hot copy)."""
    return dense_case(seed, 1, 1, 256, 256, 64, dtype="f32", hot=10.0 if hot else 1.0,
                      stream=1, name="c1_fp32_hot" if hot else "c1_fp32")


def c2_bf16(causal: bool, hot: bool = False, seed: int = BASE_SEED) -> DenseCase:
    """Batched prefill bf16: B=4, H=16, n=m=2048, d=dv=128."""
    return dense_case(seed, 4, 16, 2048, 2048, 128, dtype="bf16", causal=causal,
                      hot=10.0 if hot else 1.0, stream=2,
                      name=f"c2_bf16_{'causal' if causal else 'full'}{'_hot' if hot else ''}")


def c3_bf16(seed: int = BASE_SEED) -> DenseCase:
    """Long-context causal prefill bf16: B=1, H=32, n=m=8192, d=dv=128."""
    return dense_case(seed, 1, 32, 8192, 8192, 128, dtype="bf16", causal=True, stream=3,
                      name="c3_bf16_causal_8192")


def c4_decode(seed: int = BASE_SEED, poison: bool = True) -> DecodeCase:
    """Paged GQA decode: 64 sequences, H=32, Hkv=8, d=dv=128, page 16,
    context lengths uniform on [512, 8192]."""
    return decode_case(seed, 64, 32, 8, 128, page_size=16, len_lo=512, len_hi=8192,
                       max_blocks=512, poison=poison, stream=4)


def c5_varlen(d: int, seed: int = BASE_SEED) -> VarlenCase:
    """Ragged causal varlen prefill: 16 sequences, lengths uniform on [1, 4096],
    H=16, d=dv in {64, 128}, 10% of Q and K rows x20."""
    lens = uniform_lengths(seed, 16, 1, 4096, stream=5, tensor=9)
    return varlen_case(seed, lens, 16, d, stream=5 + d)
