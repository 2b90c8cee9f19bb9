"""Seeded synthetic inputs for paged-KV decode attention.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path and the float64 oracle consume the
arrays it returns, so the two sides always see the same fp16 bytes.

Workloads (head layouts of LLaMA-2-7B, 32x128 MHA, and LLaMA-3-8B, 32/8x128
GQA; 16-token pages):

  1  tiny GQA-2:  B=2, Hq=4, Hkv=2, D=64, L={37,100}, 32-page pool permuted,
                  q/K/V uniform in [-1, 1], no split
  2  long single sequence, MHA: B=1, 32/32, D=128, L=4096, 512-page pool
                  permuted, N(0,1)*0.5, 16 splits
  3  xLLM-style batch, MHA: B=48, 32/32, D=128, L_b = {5,13,27,51}[b%4] +
                  U{0..512}, N(0, 0.5), pages scattered
  4  GQA-4 large batch: B=160, 32/8, D=128, L_b ~ U{128..2048}, N(0, 0.5)
  5  skewed Flash-Decoding mix: B=256, 32/8, D=128, 255 x U{16..128} and one
                  32768-token sequence (last), N(0, 0.5)

Conventions (the plainest readings of the workload descriptions):
  * "N(0, s)" means standard deviation s; draws are float32, rounded to fp16
    (or, with ``dtype="bf16"``, rounded to nearest-even bf16 and kept as
    float32 arrays whose values are exactly those bf16 numbers; numpy has no
    bf16 type).  Both element types see the same draws.
  * Integer "uniform in [a, b]" is inclusive at both ends.
  * When the pool size is not given it is the pages needed plus 25 % slack,
    rounded up.  Pages come from a seeded permutation of the pool and are
    consumed in sequence order.
  * seq_lens include the token being decoded: the decode step appends k_new /
    v_new at position L_b - 1 and then attends positions 0 .. L_b - 1.
  * Pool rows that no sequence owns hold random values of the same law unless
    ``poison`` is set, in which case they hold fp16 NaN so that any read of an
    unowned row shows up in the output.
  * With ``kv="int8"`` the cache also comes as INT8 codes with one fp32 scale
    per (page, kv head, slot) row, drawn directly: codes are N(0, 40) rounded
    to integers and clipped to [-127, 127], scales uniform in [0.004, 0.012)
    (about what N(0, 0.5) rows quantise to).  Nothing here quantises; poison
    sets the scales of unowned rows to NaN.
  * With ``kv="fp8"`` the cache comes as E4M3 bytes with one fp32 scale per
    row, also drawn directly: sign uniform, exponent field e with probability
    proportional to 2^e (0 <= e <= 15, so most codes sit in the top binades,
    as rows scaled to their largest element do), mantissa uniform in 0..7,
    and the NaN pattern S.1111.111 replaced by S.1111.110; scales uniform in
    [0.001, 0.004) (about max|x| / 448 for N(0, 0.5) rows).  Poison sets the
    codes of unowned rows to the NaN pattern and their scales to NaN.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 24000
PAGE_SIZE = 16

CONFIG_NAMES = {
    1: "tiny paged decode, B=2, GQA 4/2, D=64, L={37,100}, S=16",
    2: "LLaMA-2-7B heads, B=1, MHA 32/32, D=128, L=4096, S=16, split 16",
    3: "xLLM-style batch, B=48, MHA 32/32, D=128, L={5,13,27,51}+U[0,512], S=16",
    4: "LLaMA-3-8B heads, B=160, GQA 32/8, D=128, L~U[128,2048], S=16",
    5: "skewed mix, B=256, GQA 32/8, D=128, 255xU[16,128] + 1x32768, S=16",
}


@dataclasses.dataclass
class Workload:
    """One decode step's inputs.  Arrays are host numpy arrays."""

    name: str
    config: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    max_pages_per_seq: int
    forced_splits: int          # 0 = let the planner choose
    scale: float
    seq_lens: np.ndarray        # int32 [B], includes the new token
    block_table: np.ndarray     # int32 [B][max_pages_per_seq], -1 pad
    q: np.ndarray               # fp16 [B][Hq][D]
    k_new: np.ndarray           # fp16 [B][Hkv][D]
    v_new: np.ndarray           # fp16 [B][Hkv][D]
    k_pages: np.ndarray         # fp16 [P][Hkv][S][D]
    v_pages: np.ndarray         # fp16 [P][Hkv][S][D]
    dtype: str = "fp16"                  # element type of q/K/V/out ("fp16" or "bf16")
    q_lens: np.ndarray | None = None     # int32 [B]: query tokens per sequence (multi-token);
                                         # q, k_new, v_new then have sum(q_lens) rows
    kv: str = "fp16"                     # cache format: "fp16", "int8" or "fp8"
    k_codes: np.ndarray | None = None    # [P][Hkv][S][D]: int8 codes (kv="int8") or
                                         # uint8 E4M3 bytes (kv="fp8")
    v_codes: np.ndarray | None = None
    k_scales: np.ndarray | None = None   # float32 [P][Hkv][S]
    v_scales: np.ndarray | None = None

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_bytes(self) -> int:
        """K and V bytes the step must read: sum(L) * Hkv * D * 2 tensors * 2 B."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 4

    def kv_bytes_int8(self) -> int:
        """The same for an 8-bit cache (INT8 or FP8): sum(L) * Hkv * 2 tensors * (D codes +
        a 4 B scale)."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * 2 * (self.head_dim + 4)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest-even bf16 value, returned as float32 (finite inputs)."""
    bits = np.ascontiguousarray(x, np.float32).view(np.uint32)
    bits = (bits + (np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1)))) & np.uint32(0xFFFF0000)
    return bits.view(np.float32)


def _draw(rng: np.random.Generator, shape, dist, dtype="fp16") -> np.ndarray:
    kind, param = dist
    n = int(np.prod(shape))
    if kind == "uniform":
        x = rng.random(n, dtype=np.float32) * np.float32(2.0 * param) - np.float32(param)
    elif kind == "normal":
        x = rng.standard_normal(n, dtype=np.float32) * np.float32(param)
    else:
        raise ValueError(kind)
    if dtype == "bf16":
        return round_bf16(x).reshape(shape)
    if dtype != "fp16":
        raise ValueError(dtype)
    return x.astype(np.float16).reshape(shape)


def _lengths(cfg: int, rng: np.random.Generator) -> np.ndarray:
    if cfg == 1:
        return np.array([37, 100], np.int32)
    if cfg == 2:
        return np.array([4096], np.int32)
    if cfg == 3:
        prompt = np.array([5, 13, 27, 51], np.int32)[np.arange(48) % 4]
        return (prompt + rng.integers(0, 512, size=48, endpoint=True)).astype(np.int32)
    if cfg == 4:
        return rng.integers(128, 2048, size=160, endpoint=True).astype(np.int32)
    if cfg == 5:
        short = rng.integers(16, 128, size=255, endpoint=True)
        return np.concatenate([short, [32768]]).astype(np.int32)
    raise ValueError(f"unknown config {cfg}")


_SHAPES = {
    # cfg: (Hq, Hkv, D, pool pages or None, distribution, forced splits)
    1: (4, 2, 64, 32, ("uniform", 1.0), 1),
    2: (32, 32, 128, 512, ("normal", 0.5), 16),
    3: (32, 32, 128, None, ("normal", 0.5), 0),
    4: (32, 8, 128, None, ("normal", 0.5), 0),
    5: (32, 8, 128, None, ("normal", 0.5), 0),
}


def layout(seq_lens: np.ndarray, num_pages: int, page_size: int, rng: np.random.Generator,
           max_pages_per_seq: int | None = None) -> np.ndarray:
    """Block table from a seeded permutation of the pool, consumed in sequence order."""
    pages_needed = [(int(l) + page_size - 1) // page_size for l in seq_lens]
    width = max(max(pages_needed, default=0), 1) if max_pages_per_seq is None else max_pages_per_seq
    if sum(pages_needed) > num_pages:
        raise ValueError("pool too small")
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(seq_lens), width), -1, np.int32)
    cursor = 0
    for b, n in enumerate(pages_needed):
        bt[b, :n] = perm[cursor:cursor + n]
        cursor += n
    return bt


def make_custom(*, seq_lens, num_q_heads, num_kv_heads, head_dim, page_size=PAGE_SIZE,
                num_pages=None, dist=("normal", 0.5), seed=0, forced_splits=0,
                scale=None, poison=False, max_pages_per_seq=None, name="custom",
                config=0, kv="fp16", dtype="fp16", q_lens=None) -> Workload:
    """Any shape: used by the tests for ragged, empty and edge cases.  With
    ``q_lens`` the step has q_lens[b] query tokens per sequence (the newest
    ones, q_lens[b] <= seq_lens[b]), packed sequence after sequence."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    B = len(seq_lens)
    needed = sum((int(l) + page_size - 1) // page_size for l in seq_lens)
    if num_pages is None:
        num_pages = max(1, math.ceil(needed * 1.25))
    bt = layout(seq_lens, num_pages, page_size, rng, max_pages_per_seq)
    rows = B
    if q_lens is not None:
        q_lens = np.asarray(q_lens, np.int32)
        if len(q_lens) != B or np.any(q_lens < 0) or np.any(q_lens > seq_lens):
            raise ValueError("need 0 <= q_lens[b] <= seq_lens[b]")
        rows = int(q_lens.sum())
    q = _draw(rng, (rows, num_q_heads, head_dim), dist, dtype)
    k_new = _draw(rng, (rows, num_kv_heads, head_dim), dist, dtype)
    v_new = _draw(rng, (rows, num_kv_heads, head_dim), dist, dtype)
    pool_shape = (num_pages, num_kv_heads, page_size, head_dim)
    k_pages = _draw(rng, pool_shape, dist, dtype)
    v_pages = _draw(rng, pool_shape, dist, dtype)
    if poison:
        owned = np.zeros((num_pages, page_size), bool)
        for b, L in enumerate(seq_lens):
            for t in range(int(L)):
                owned[bt[b, t // page_size], t % page_size] = True
        pg, slot = np.nonzero(~owned)
        k_pages[pg, :, slot, :] = np.nan
        v_pages[pg, :, slot, :] = np.nan
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    q8 = {}
    if kv == "int8":
        def codes():
            c = np.rint(rng.standard_normal(pool_shape, dtype=np.float32) * np.float32(40.0))
            return np.clip(c, -127, 127).astype(np.int8)

        def scales():
            return (np.float32(0.004) + rng.random(pool_shape[:3], dtype=np.float32)
                    * np.float32(0.008)).astype(np.float32)

        q8 = dict(k_codes=codes(), v_codes=codes(), k_scales=scales(), v_scales=scales())
        if poison:
            q8["k_scales"][pg, :, slot] = np.float32(np.nan)
            q8["v_scales"][pg, :, slot] = np.float32(np.nan)
    elif kv == "fp8":
        pe = np.exp2(np.arange(16, dtype=np.float64))
        pe /= pe.sum()

        def codes():
            sign = rng.integers(0, 2, size=pool_shape, dtype=np.uint8) << 7
            e = rng.choice(16, size=pool_shape, p=pe).astype(np.uint8)
            m = rng.integers(0, 8, size=pool_shape, dtype=np.uint8)
            c = sign | (e << 3) | m
            return np.where((c & 0x7F) == 0x7F, c - 1, c).astype(np.uint8)

        def scales():
            return (np.float32(0.001) + rng.random(pool_shape[:3], dtype=np.float32)
                    * np.float32(0.003)).astype(np.float32)

        q8 = dict(k_codes=codes(), v_codes=codes(), k_scales=scales(), v_scales=scales())
        if poison:
            for key in ("k_codes", "v_codes"):
                q8[key][pg, :, slot, :] = np.uint8(0x7F)
            q8["k_scales"][pg, :, slot] = np.float32(np.nan)
            q8["v_scales"][pg, :, slot] = np.float32(np.nan)
    elif kv != "fp16":
        raise ValueError(kv)
    return Workload(name=name, config=config, batch=B, num_q_heads=num_q_heads,
                    num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size,
                    num_pages=num_pages, max_pages_per_seq=bt.shape[1],
                    forced_splits=forced_splits, scale=float(scale), seq_lens=seq_lens,
                    block_table=bt, q=q, k_new=k_new, v_new=v_new, k_pages=k_pages,
                    v_pages=v_pages, dtype=dtype, q_lens=q_lens, kv=kv, **q8)


def make_config(cfg: int, seed: int | None = None, poison: bool = False,
                kv: str = "fp16", dtype: str = "fp16") -> Workload:
    """The five benchmark workloads, seeded with 24000 + cfg by default."""
    if cfg not in _SHAPES:
        raise ValueError(f"unknown config {cfg}")
    seed = SEED_BASE + cfg if seed is None else seed
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, pool, dist, splits = _SHAPES[cfg]
    seq_lens = _lengths(cfg, rng)
    # The remaining draws come from a second stream so that the lengths above
    # do not shift when the pool size changes.
    sub_seed = int(rng.integers(0, 2**31 - 1))
    w = make_custom(seq_lens=seq_lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                    page_size=PAGE_SIZE, num_pages=pool, dist=dist, seed=sub_seed,
                    forced_splits=splits, poison=poison, name=CONFIG_NAMES[cfg], config=cfg,
                    kv=kv, dtype=dtype)
    return w


PREFILL_NAMES = {
    1: "chunked prefill, LLaMA-3-8B heads: B=16, GQA 32/8, D=128, L~U[1024,4096], last 512 "
       "tokens queried",
    2: "piggybacked prefill + decode, LLaMA-3-8B heads: 8 prefill chunks of 256 at L~U[256,2048] "
       "and 56 decode tokens at L~U[128,2048], GQA 32/8, D=128",
}


def make_prefill_config(cfg: int, seed: int | None = None, dtype: str = "fp16") -> Workload:
    """Multi-token workloads (several query tokens per sequence), seeded
    with 24100 + cfg by default.  Query tokens are the newest of their
    sequence; values N(0, 0.5) as in the decode workloads."""
    seed = SEED_BASE + 100 + cfg if seed is None else seed
    rng = np.random.default_rng(seed)
    if cfg == 1:
        lens = rng.integers(1024, 4096, size=16, endpoint=True).astype(np.int32)
        q_lens = np.full(16, 512, np.int32)
    elif cfg == 2:
        pre = rng.integers(256, 2048, size=8, endpoint=True)
        dec = rng.integers(128, 2048, size=56, endpoint=True)
        lens = np.concatenate([pre, dec]).astype(np.int32)
        q_lens = np.concatenate([np.full(8, 256), np.ones(56)]).astype(np.int32)
    else:
        raise ValueError(f"unknown multi-token workload {cfg}")
    sub_seed = int(rng.integers(0, 2**31 - 1))
    return make_custom(seq_lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128,
                       dist=("normal", 0.5), seed=sub_seed, q_lens=q_lens,
                       name=PREFILL_NAMES[cfg], config=cfg, dtype=dtype)

