"""Seeded synthetic inputs for the NVFP4 paged KV-cache path.

This module draws random numbers and lays out page tables; it holds none of
the method's arithmetic (no quantisation, no attention).  Both the CUDA path
(tests, bench) and the CPU oracle take their inputs from here, so the two see
exactly the same values.

The pages measure serving runs with real prompts and model weights that are
not available here; these generators reproduce only the shapes, lengths, value
distributions and residency counts of those workloads:

  tiny      1 layer, batch 2, Hq=8, Hkv=2, d=128, 256 tokens per sequence,
            page 16, shuffled page table; K/V ~ N(0,1); query bf16 N(0,1).
  llama70b  Llama-3.3-70B-shaped layer: Hq=64, Hkv=8, d=128, batch 12 or 21 at
            8192 tokens; per kv head 4 of 128 channels scaled x10 (the same
            channels for K and V); bf16 query.
  ctx32k    Hq=48, Hkv=8, batch 44 or 70, lengths uniform in [24576, 32768];
            every (K or V, kv head) scaled by a factor uniform in [0.5, 4].
  ctx160k   Hq=48, Hkv=8, batch 10 or 15 at 163840 tokens; K/V ~ N(0,1).
  ctx1m     Hq=48, Hkv=8, batch 1 or 2 at 1048576 tokens; per kv head 4 of 128
            channels drawn from Student-t(3) instead of N(0,1).

Values are generated in fixed chunks of CHUNK tokens per (sequence, K|V) from
a generator seeded by (workload seed, K|V, sequence, chunk), so any slice can
be regenerated on its own.  torch's CPU and CUDA generators give different
streams: callers that compare devices generate once and copy.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np
import torch

CHUNK = 4096
HEAD_DIM = 128
PAGE_SIZE = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    seq_lens: tuple
    seed: int
    dist: str                     # normal | outlier10 | headscale | student_t
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    input_dtype: str = "f32"      # dtype of the new K/V rows fed to quantize_append

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def pages_per_seq(self) -> list:
        P = self.page_size
        return [(L + P - 1) // P for L in self.seq_lens]

    @property
    def max_pages(self) -> int:
        return max(1, max(self.pages_per_seq))

    @property
    def num_pages(self) -> int:
        return max(1, sum(self.pages_per_seq))

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens))


def _seed(*parts) -> int:
    # integers of any type (Python or numpy) seed identically
    norm = tuple(int(x) if isinstance(x, (int, np.integer)) else x for x in parts)
    return zlib.crc32(repr(norm).encode()) & 0x7FFFFFFF


def make(name: str, batch: int | None = None, seq_len: int | None = None) -> Workload:
    """The five workloads; ``batch``/``seq_len`` override the default sizes."""
    if name == "tiny":
        B = batch or 2
        L = seq_len or 256
        return Workload(name, B, 8, 2, tuple([L] * B), 0, "normal")
    if name == "llama70b":
        B = batch or 12
        L = seq_len or 8192
        return Workload(name, B, 64, 8, tuple([L] * B), 1, "outlier10")
    if name == "ctx32k":
        B = batch or 44
        rng = np.random.default_rng(_seed(2, "lens", B))
        lo, hi = 24576, 32768
        if seq_len is not None:
            lo, hi = max(1, seq_len * 3 // 4), seq_len
        lens = tuple(int(v) for v in rng.integers(lo, hi + 1, size=B))
        return Workload(name, B, 48, 8, lens, 2, "headscale")
    if name == "ctx160k":
        B = batch or 10
        L = seq_len or 163840
        return Workload(name, B, 48, 8, tuple([L] * B), 3, "normal", input_dtype="bf16")
    if name == "ctx1m":
        B = batch or 1
        L = seq_len or 1048576
        return Workload(name, B, 48, 8, tuple([L] * B), 4, "student_t")
    raise ValueError(f"unknown workload {name!r}")


def custom(batch, num_q_heads, num_kv_heads, seq_lens, seed=7, dist="normal") -> Workload:
    return Workload("custom", batch, num_q_heads, num_kv_heads, tuple(int(x) for x in seq_lens),
                    seed, dist)


def block_table(w: Workload, pad_value: int = -1, spare_pages: int = 0):
    """A random permutation of physical pages handed out to the sequences in order.

    Returns (block_table int32 [B][max_pages], num_pages).  Entries past a
    sequence's last page hold ``pad_value``; ``spare_pages`` unused pages are
    added to the pool so the table is not a bijection onto it.
    """
    num_pages = w.num_pages + spare_pages
    rng = np.random.default_rng(_seed(w.seed, "pages", w.batch))
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((w.batch, w.max_pages), pad_value, np.int32)
    off = 0
    for b, n in enumerate(w.pages_per_seq):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, num_pages


def slot_mapping(w: Workload, bt: np.ndarray, b: int, t0: int, t1: int) -> np.ndarray:
    """Cache slots (page * page_size + offset) of tokens t0..t1-1 of sequence b."""
    j = np.arange(t0, t1)
    P = w.page_size
    return (bt[b, j // P].astype(np.int64) * P + j % P).astype(np.int32)


def _channel_mods(w: Workload):
    """Per-kv-head channel choices and scales that shape the K/V distribution."""
    rng = np.random.default_rng(_seed(w.seed, "mods"))
    Hkv, d = w.num_kv_heads, w.head_dim
    special = np.stack([rng.choice(d, size=4, replace=False) for _ in range(Hkv)])
    head_scale = rng.uniform(0.5, 4.0, size=(2, Hkv))          # [K|V][Hkv]
    return special, head_scale


def _chunk(w: Workload, which: int, b: int, c: int, device) -> torch.Tensor:
    L = w.seq_lens[b]
    t0 = c * CHUNK
    n = min(CHUNK, L - t0)
    gen = torch.Generator(device=device)
    gen.manual_seed(_seed(w.seed, which, b, c))
    x = torch.randn((n, w.num_kv_heads, w.head_dim), generator=gen, device=device,
                    dtype=torch.float32)
    if w.dist == "normal":
        return x
    special, head_scale = _channel_mods(w)
    if w.dist == "outlier10":
        for h in range(w.num_kv_heads):
            x[:, h, torch.as_tensor(special[h], device=device)] *= 10.0
    elif w.dist == "headscale":
        hs = torch.as_tensor(head_scale[which], dtype=torch.float32, device=device)
        x *= hs.view(1, -1, 1)
    elif w.dist == "student_t":
        z = torch.randn((n, w.num_kv_heads, 4), generator=gen, device=device)
        chi = torch.randn((n, w.num_kv_heads, 4, 3), generator=gen, device=device)
        t = z / torch.sqrt((chi * chi).sum(-1) / 3.0)
        for h in range(w.num_kv_heads):
            x[:, h, torch.as_tensor(special[h], device=device)] = t[:, h]
    else:
        raise ValueError(w.dist)
    return x


def kv_rows(w: Workload, which: str, b: int, t0: int, t1: int, device="cpu") -> torch.Tensor:
    """fp32 K (which='k') or V ('v') rows [t1-t0][Hkv][d] of sequence b."""
    wi = {"k": 0, "v": 1}[which]
    parts = []
    c0, c1 = t0 // CHUNK, (t1 - 1) // CHUNK
    for c in range(c0, c1 + 1):
        x = _chunk(w, wi, b, c, device)
        lo = max(t0 - c * CHUNK, 0)
        hi = min(t1 - c * CHUNK, x.shape[0])
        parts.append(x[lo:hi])
    return torch.cat(parts, 0) if len(parts) > 1 else parts[0]


def query(w: Workload, device="cpu") -> torch.Tensor:
    """bf16 queries [B][Hq][d] ~ N(0,1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(_seed(w.seed, "q", w.batch))
    q = torch.randn((w.batch, w.num_q_heads, w.head_dim), generator=gen, device=device)
    return q.to(torch.bfloat16)


def new_tokens(w: Workload, T: int, device="cpu", salt: str = "new"):
    """fp32 K and V rows [T][Hkv][d] for appending T fresh tokens."""
    gen = torch.Generator(device=device)
    gen.manual_seed(_seed(w.seed, salt, T))
    k = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen, device=device)
    v = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen, device=device)
    return k, v


# --- extend path -------------------------------------------------------------
#
# The extend step attends a chunk of new tokens over its sequence's prefix,
# held in the FP8 workspace, and over the chunk itself.  Inputs: bf16 queries
# and chunk K/V ~ N(0,1); workspace rows of random finite E4M3 codes (sign
# random, exponent field uniform in 1..8, mantissa uniform, 1 in 32 zero), i.e.
# magnitudes log-uniform in [2^-6, 3.75].  Sequences sit in the workspace with
# EXTEND_GAP unused rows before each, so their row offsets are not contiguous.

EXTEND_GAP = 3


@dataclasses.dataclass(frozen=True)
class ExtendWorkload:
    name: str
    prefix_lens: tuple
    chunk_lens: tuple
    num_q_heads: int
    num_kv_heads: int
    seed: int
    head_dim: int = HEAD_DIM

    @property
    def batch(self) -> int:
        return len(self.prefix_lens)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def q_rows(self) -> int:
        return int(sum(self.chunk_lens))

    @property
    def prefix_rows(self) -> int:
        return int(sum(self.prefix_lens)) + EXTEND_GAP * (self.batch + 1)

    def q_indptr(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk_lens)]).astype(np.int32)

    def kv_indptr(self) -> np.ndarray:
        starts = EXTEND_GAP * np.arange(1, self.batch + 1) + np.concatenate([[0], np.cumsum(self.prefix_lens)[:-1]])
        return starts.astype(np.int32)


def extend_make(name: str) -> ExtendWorkload:
    """ext160k: the last 8,192-token chunk of a 163,840-token prefill (Hq=48,
    Hkv=8), prefix 155,648.  ext8k_c2k: a 2,048-token chunk over an 8,192-token
    prefix (the profiling case).  ext_small: four ragged sequences.
    prefill8k: initial prefill of one 8,192-token prompt (no prefix; Hq=48,
    Hkv=8), the chunk the 160K workload quantises."""
    if name == "prefill8k":
        return ExtendWorkload(name, (0,), (8192,), 48, 8, seed=_seed("prefill8k"))
    if name == "ext160k":
        return ExtendWorkload(name, (163840 - 8192,), (8192,), 48, 8, seed=_seed("ext160k"))
    if name == "ext8k_c2k":
        return ExtendWorkload(name, (8192,), (2048,), 48, 8, seed=_seed("ext8k_c2k"))
    if name == "ext_small":
        return ExtendWorkload(name, (0, 61, 200, 1000), (130, 1, 77, 64), 48, 8, seed=_seed("ext_small"))
    raise ValueError(name)


def extend_custom(prefix_lens, chunk_lens, num_q_heads, num_kv_heads, seed=11) -> ExtendWorkload:
    return ExtendWorkload("custom", tuple(int(x) for x in prefix_lens), tuple(int(x) for x in chunk_lens),
                          num_q_heads, num_kv_heads, seed=seed)


def e4m3_codes(shape, gen, device="cpu") -> torch.Tensor:
    """Random finite E4M3 bytes as described above (uint8)."""
    e = torch.randint(1, 9, shape, generator=gen, device=device, dtype=torch.int32)
    m = torch.randint(0, 8, shape, generator=gen, device=device, dtype=torch.int32)
    s = torch.randint(0, 2, shape, generator=gen, device=device, dtype=torch.int32)
    z = torch.randint(0, 32, shape, generator=gen, device=device, dtype=torch.int32) == 0
    code = (s << 7) | (e << 3) | m
    return torch.where(z, torch.zeros_like(code), code).to(torch.uint8)


def extend_inputs(e: ExtendWorkload, device="cpu", chunk: str = "bf16") -> dict:
    """q (bf16 [rows][Hq][d]), k_chunk / v_chunk ([rows][Hkv][d]: bf16 ~ N(0,1),
    or with chunk="e4m3" random E4M3 codes as uint8, the prompt's K/V as FP8),
    k_prefix / v_prefix (uint8 E4M3 [prefix rows][Hkv][d]) and the int32 index
    arrays q_indptr, kv_indptr, prefix_lens."""
    gen = torch.Generator(device=device)
    gen.manual_seed(_seed(e.seed, "extend"))
    rows, d = e.q_rows, e.head_dim
    q = torch.randn((rows, e.num_q_heads, d), generator=gen, device=device).to(torch.bfloat16)
    if chunk == "bf16":
        kc = torch.randn((rows, e.num_kv_heads, d), generator=gen, device=device).to(torch.bfloat16)
        vc = torch.randn((rows, e.num_kv_heads, d), generator=gen, device=device).to(torch.bfloat16)
    elif chunk == "e4m3":
        kc = e4m3_codes((rows, e.num_kv_heads, d), gen, device)
        vc = e4m3_codes((rows, e.num_kv_heads, d), gen, device)
    else:
        raise ValueError(chunk)
    out = {
        "q": q,
        "k_chunk": kc,
        "v_chunk": vc,
        "k_prefix": e4m3_codes((e.prefix_rows, e.num_kv_heads, d), gen, device),
        "v_prefix": e4m3_codes((e.prefix_rows, e.num_kv_heads, d), gen, device),
    }
    for k, v in (("q_indptr", e.q_indptr()), ("kv_indptr", e.kv_indptr()),
                 ("prefix_lens", np.asarray(e.prefix_lens, np.int32))):
        out[k] = torch.from_numpy(v).to(device)
    return out
