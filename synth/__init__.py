"""Seeded synthetic inputs for paged FP8 attention.

This module draws the inputs that both the CUDA library and the CPU oracle
consume.  It holds none of the attention arithmetic: it only draws random
numbers, lays out 64-token pages behind a randomly permuted block table, and
turns K/V into E4M3 bytes with torch's own float8_e4m3fn conversion (the K/V
bytes are inputs; the oracle decodes them, the kernels read them).

Recipe (shared by every workload):
  * Q: bf16 N(0, 1).  q_descale = amax|q| / 448 (fp32).
  * K, V: N(0, 1), then max(1, round(0.01 * D)) channels per KV head (drawn
    per tensor from the seeded generator) multiplied by 8; per-tensor
    descale = amax / 448; bytes = e4m3(x / descale).
  * Pages: every logical page a sequence can see maps to its own physical page,
    in a random permutation.  Pages no query of the sequence can see map to one
    shared poison page whose bytes are 0x7F (E4M3 NaN), and the slots of a last
    page that lie at or beyond the sequence length hold 0x7F as well, so any
    read outside the visible set turns the output into NaN.
  * softmax_scale = 1 / sqrt(D).

Named workloads follow the five benchmark configurations: a tiny causal
prefill, a sliding-window decode at head dim 256, a full-attention decode at
head dim 512 (BF16 Q, and FP8 Q), a chunked-prefill mixed batch (head dim 256
with a 1024-key window; head dim 512 causal) and a speculative-verify batch
whose 25600-token prefix pages are shared by all sequences.

The KV-cache write workloads draw the new keys and values of the mixed batch's
8128 tokens with the same K/V recipe (bf16 here, before any quantization), and
a slot mapping: the chunk's 4096 tokens fill 64 whole pages, and each decode
token takes the next row of its own sequence's last page (a random row of its
own page).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

PAGE = 64
POISON = 0x7F


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor             # bf16 [total_q, Hq, D]
    q_descale: float
    k_cache: torch.Tensor       # uint8 [num_pages, 64, Hkv, D]
    v_cache: torch.Tensor
    k_descale: float
    v_descale: float
    block_table: torch.Tensor   # int32 [B, max_pages_per_seq]
    cu_seqlens_q: torch.Tensor  # int32 [B + 1]
    seqused_k: torch.Tensor     # int32 [B]
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    softmax_scale: float
    window_left: int
    causal: bool
    fp8_q: bool                 # FP8-MMA path (Q quantized to E4M3) or BF16-Q path
    lq: np.ndarray              # host copies of the structure
    lk: np.ndarray
    bt: np.ndarray
    poison_page: int
    seed: int
    v_channel_scale: np.ndarray  # [Hkv, D]: 1 or 8, the scale each V channel was drawn with

    @property
    def batch(self) -> int:
        return int(self.lq.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.lq.sum())

    @property
    def max_seqlen_q(self) -> int:
        return int(self.lq.max()) if self.lq.size else 0

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    def visible_pairs(self) -> int:
        """Number of (query row, key) pairs that are visible, summed over heads
        of one KV-head group: sum over queries of |J|, times Hq."""
        return int(sum(_visible_count(int(a), int(b), self.window_left, self.causal)
                       for a, b in zip(self.lq, self.lk))) * self.num_heads_q

    def kv_bytes_algorithmic(self) -> int:
        """K+V bytes of every (sequence, KV head) visible key set: a key that any
        query of the sequence sees counts once per KV head, D bytes for K and
        D for V."""
        keys = 0
        for a, b in zip(self.lq, self.lk):
            rng = _seq_visible_span(int(a), int(b), self.window_left, self.causal)
            if rng is not None:
                keys += rng[1] - rng[0] + 1
        return keys * self.num_heads_kv * self.head_dim * 2

    def flops_algorithmic(self) -> int:
        """QK^T + PV flops over visible pairs only: 4 * D per (query, head, key)."""
        return self.visible_pairs() * 4 * self.head_dim


def _visible_count(Lq: int, Lk: int, window_left: int, causal: bool) -> int:
    n = 0
    for i in range(Lq):
        p = Lk - Lq + i
        lo = max(0, p - window_left) if window_left >= 0 else 0
        hi = min(p, Lk - 1) if causal else Lk - 1
        if Lk > 0 and hi >= lo:
            n += hi - lo + 1
    return n


def _seq_visible_span(Lq: int, Lk: int, window_left: int, causal: bool):
    """[lo, hi] union of the visible key ranges of a sequence's queries (None if empty)."""
    if Lq <= 0 or Lk <= 0:
        return None
    p0 = Lk - Lq
    lo = max(0, p0 - window_left) if window_left >= 0 else 0
    pl = Lk - 1
    hi = min(pl, Lk - 1) if causal else Lk - 1
    if causal and p0 + (Lq - 1) < 0:
        return None
    if hi < lo:
        return None
    # first query may see nothing under causal when p < 0; the union is still [lo, hi]
    return lo, hi


def _torch_gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7_919 + 12_345) % (2**63 - 1))
    return g


def build_structure(lq: Sequence[int], lk: Sequence[int], window_left: int, causal: bool, seed: int,
                    shared_prefix_pages: int = 0):
    """Block table and physical page count.

    Returns (block_table [B, max_pages] int32, num_phys_pages, poison_page,
    tail_slots) where tail_slots lists (phys_page, first_poison_slot) for last
    pages that end before slot 64."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    lq = np.asarray(lq, dtype=np.int64)
    lk = np.asarray(lk, dtype=np.int64)
    B = lq.shape[0]
    pages_per_seq = (lk + PAGE - 1) // PAGE
    max_pages = max(1, int(pages_per_seq.max()) if B else 1)
    # logical pages that need their own storage
    need = []  # (b, j)
    for b in range(B):
        span = _seq_visible_span(int(lq[b]), int(lk[b]), window_left, causal)
        if span is None:
            continue
        j0, j1 = span[0] // PAGE, span[1] // PAGE
        for j in range(j0, j1 + 1):
            if j < shared_prefix_pages:
                continue
            need.append((b, j))
    n_phys = 1 + shared_prefix_pages + len(need)
    perm = rng.permutation(n_phys).astype(np.int64)
    poison_page = int(perm[0])
    shared_ids = perm[1:1 + shared_prefix_pages]
    bt = np.full((B, max_pages), poison_page, dtype=np.int32)
    for b in range(B):
        npg = int(pages_per_seq[b])
        for j in range(min(shared_prefix_pages, npg)):
            bt[b, j] = shared_ids[j]
    tail = []
    for idx, (b, j) in enumerate(need):
        phys = int(perm[1 + shared_prefix_pages + idx])
        bt[b, j] = phys
    for b in range(B):
        L = int(lk[b])
        if L % PAGE and L > 0:
            j = (L - 1) // PAGE
            if bt[b, j] != poison_page:
                tail.append((int(bt[b, j]), L % PAGE))
    return bt, n_phys, poison_page, tail


def _channel_scale(rng: np.random.Generator, hkv: int, d: int) -> np.ndarray:
    s = np.ones((hkv, d), dtype=np.float32)
    n = max(1, int(round(0.01 * d)))
    for h in range(hkv):
        idx = rng.choice(d, size=n, replace=False)
        s[h, idx] = 8.0
    return s


def _fill_cache(n_phys: int, hkv: int, d: int, scale: np.ndarray, seed: int, stream: int, device,
                chunk_pages: int):
    """Two passes over seeded chunks: amax, then quantize.  Returns (cache uint8, descale)."""
    sc = torch.from_numpy(scale).to(device)
    amax = torch.zeros((), dtype=torch.float32, device=device)
    n_chunks = (n_phys + chunk_pages - 1) // chunk_pages
    for c in range(n_chunks):
        p0, p1 = c * chunk_pages, min(n_phys, (c + 1) * chunk_pages)
        g = _torch_gen(device, seed, stream * 1_000_000 + c)
        x = torch.randn((p1 - p0, PAGE, hkv, d), generator=g, device=device, dtype=torch.float32) * sc
        amax = torch.maximum(amax, x.abs().amax())
        del x
    descale = float(amax.item()) / 448.0
    descale = float(np.float32(np.float32(amax.item()) / np.float32(448.0)))
    cache = torch.empty((n_phys, PAGE, hkv, d), dtype=torch.uint8, device=device)
    for c in range(n_chunks):
        p0, p1 = c * chunk_pages, min(n_phys, (c + 1) * chunk_pages)
        g = _torch_gen(device, seed, stream * 1_000_000 + c)
        x = torch.randn((p1 - p0, PAGE, hkv, d), generator=g, device=device, dtype=torch.float32) * sc
        cache[p0:p1] = (x / descale).to(torch.float8_e4m3fn).view(torch.uint8)
        del x
    return cache, descale


def make_workload(name: str, lq: Sequence[int], lk: Sequence[int], num_heads_q: int, num_heads_kv: int,
                  head_dim: int, window_left: int, causal: bool, fp8_q: bool, seed: int, device="cpu",
                  shared_prefix_pages: int = 0, chunk_pages: Optional[int] = None) -> Workload:
    lq = np.asarray(lq, dtype=np.int32)
    lk = np.asarray(lk, dtype=np.int32)
    bt, n_phys, poison_page, tail = build_structure(lq, lk, window_left, causal, seed, shared_prefix_pages)
    rng = np.random.default_rng(np.random.PCG64(seed + 17))
    k_scale = _channel_scale(rng, num_heads_kv, head_dim)
    v_scale = _channel_scale(rng, num_heads_kv, head_dim)
    if chunk_pages is None:
        per_page = PAGE * num_heads_kv * head_dim * 4
        chunk_pages = max(1, (256 << 20) // per_page)
    k_cache, k_descale = _fill_cache(n_phys, num_heads_kv, head_dim, k_scale, seed, 1, device, chunk_pages)
    v_cache, v_descale = _fill_cache(n_phys, num_heads_kv, head_dim, v_scale, seed, 2, device, chunk_pages)
    k_cache[poison_page] = POISON
    v_cache[poison_page] = POISON
    for phys, first in tail:
        k_cache[phys, first:] = POISON
        v_cache[phys, first:] = POISON
    total_q = int(lq.sum())
    g = _torch_gen(device, seed, 3)
    q = torch.randn((total_q, num_heads_q, head_dim), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    qa = float(q.float().abs().amax().item()) if total_q else 1.0
    q_descale = float(np.float32(np.float32(qa) / np.float32(448.0)))
    cu = np.zeros((lq.shape[0] + 1,), dtype=np.int32)
    cu[1:] = np.cumsum(lq)
    return Workload(
        name=name, q=q, q_descale=q_descale, k_cache=k_cache, v_cache=v_cache, k_descale=k_descale,
        v_descale=v_descale, block_table=torch.from_numpy(bt).to(device),
        cu_seqlens_q=torch.from_numpy(cu).to(device), seqused_k=torch.from_numpy(lk.copy()).to(device),
        num_heads_q=num_heads_q, num_heads_kv=num_heads_kv, head_dim=head_dim,
        softmax_scale=float(np.float32(1.0 / math.sqrt(head_dim))), window_left=window_left, causal=causal,
        fp8_q=fp8_q, lq=lq, lk=lk, bt=bt, poison_page=poison_page, seed=seed, v_channel_scale=v_scale)


# ------------------------------------------------------------------ named workloads

CONFIG_NAMES = [
    "tiny_prefill_hd256",          # 2 seqs (96, 160), causal, Hq 4 / Hkv 2, D 256, FP8 Q
    "swa_decode_hd256",            # 64 x 1 query, Lk ~ U[1024, 9216], window 1023, Hq 32 / Hkv 16, FP8 Q
    "full_decode_hd512_bf16q",     # 64 x 1 query, Lk ~ U[8192, 9216], Hq 32 / Hkv 4, D 512, BF16 Q
    "full_decode_hd512_fp8q",      # same inputs, Q quantized to E4M3 (FP8-MMA path)
    "mixed_hd256_swa",             # 4096-token chunk on 4096 cached + 4032 decodes, window 1023, FP8 Q
    "mixed_hd512_causal",          # same batch, D 512 causal, Hq 32 / Hkv 4, BF16 Q
    "mixed_hd512_causal_fp8q",     # same batch, FP8 Q
    "spec_verify_hd512",           # 64 x 4 causal queries, 25600 shared + 3072 unique keys, BF16 Q
    "chunk_hd256_swa",             # the mixed batch's 4096-token chunk alone (prefill, tensor-bound)
    "chunk_hd512_causal",
    "chunk_hd512_causal_fp8q",
]


def make_config(name: str, device="cpu", scale_batch: float = 1.0) -> Workload:
    """Build a named workload.  scale_batch < 1 keeps the per-sequence shapes and
    draws fewer sequences (used by tests that need a smaller instance)."""
    def nb(b):
        return max(1, int(round(b * scale_batch)))

    if name == "tiny_prefill_hd256":
        return make_workload(name, [96, 160], [96, 160], 4, 2, 256, -1, True, True, seed=0, device=device)
    if name == "swa_decode_hd256":
        rng = np.random.default_rng(np.random.PCG64(1001))
        B = nb(64)
        lk = rng.integers(1024, 9216 + 1, size=B)
        return make_workload(name, [1] * B, lk, 32, 16, 256, 1023, True, True, seed=1, device=device)
    if name in ("full_decode_hd512_bf16q", "full_decode_hd512_fp8q"):
        rng = np.random.default_rng(np.random.PCG64(1002))
        B = nb(64)
        lk = rng.integers(8192, 9216 + 1, size=B)
        return make_workload(name, [1] * B, lk, 32, 4, 512, -1, True, name.endswith("fp8q"), seed=2,
                             device=device)
    if name in ("mixed_hd256_swa", "mixed_hd512_causal", "mixed_hd512_causal_fp8q"):
        rng = np.random.default_rng(np.random.PCG64(1003))
        nd = nb(4032)
        lk = np.concatenate([[8192], rng.integers(512, 8192 + 1, size=nd)])
        lq = np.concatenate([[4096], np.ones(nd, dtype=np.int64)])
        if name == "mixed_hd256_swa":
            return make_workload(name, lq, lk, 32, 16, 256, 1023, True, True, seed=3, device=device)
        return make_workload(name, lq, lk, 32, 4, 512, -1, True, name.endswith("fp8q"), seed=3, device=device)
    if name == "chunk_hd256_swa":
        return make_workload(name, [4096], [8192], 32, 16, 256, 1023, True, True, seed=3, device=device)
    if name in ("chunk_hd512_causal", "chunk_hd512_causal_fp8q"):
        return make_workload(name, [4096], [8192], 32, 4, 512, -1, True, name.endswith("fp8q"), seed=3,
                             device=device)
    if name == "spec_verify_hd512":
        B = nb(64)
        lk = [25600 + 3072] * B
        return make_workload(name, [4] * B, lk, 32, 4, 512, -1, True, False, seed=4, device=device,
                             shared_prefix_pages=25600 // PAGE)
    raise KeyError(name)


def subproblem_pages(w: Workload, seqs: Sequence[int]):
    """Host (numpy) copy of just the pages that sequences `seqs` reference, with
    a remapped block table.  Returns dict with q (bf16 bits, uint16), k, v,
    block_table, cu_seqlens_q, seqused_k and the token offset map."""
    seqs = [int(s) for s in seqs]
    bt = w.bt[seqs]
    pages_used = (w.lk[seqs].astype(np.int64) + PAGE - 1) // PAGE
    phys = sorted({int(bt[i, j]) for i in range(len(seqs)) for j in range(int(pages_used[i]))})
    remap = {p: i for i, p in enumerate(phys)}
    idx = torch.tensor(phys, dtype=torch.long, device=w.k_cache.device)
    k = w.k_cache.index_select(0, idx).cpu().numpy() if phys else np.zeros((0, PAGE, w.num_heads_kv, w.head_dim), np.uint8)
    v = w.v_cache.index_select(0, idx).cpu().numpy() if phys else np.zeros_like(k)
    nbt = np.zeros((len(seqs), max(1, bt.shape[1])), dtype=np.int32)
    for i in range(len(seqs)):
        for j in range(int(pages_used[i])):
            nbt[i, j] = remap[int(bt[i, j])]
    cu_full = np.zeros((w.batch + 1,), dtype=np.int64)
    cu_full[1:] = np.cumsum(w.lq)
    tok = []
    for s in seqs:
        tok.extend(range(int(cu_full[s]), int(cu_full[s + 1])))
    tok_t = torch.tensor(tok, dtype=torch.long, device=w.q.device)
    q = w.q.index_select(0, tok_t).cpu().view(torch.int16).numpy().view(np.uint16) if tok else \
        np.zeros((0, w.num_heads_q, w.head_dim), np.uint16)
    lq = w.lq[seqs]
    cu = np.zeros((len(seqs) + 1,), dtype=np.int32)
    cu[1:] = np.cumsum(lq)
    return dict(q=q, k=k, v=v, block_table=nbt, cu_seqlens_q=cu, seqused_k=w.lk[seqs].astype(np.int32),
                tokens=np.asarray(tok, dtype=np.int64))


# ------------------------------------------------------------------ KV-cache write inputs

def kv_like_values(T: int, hkv: int, d: int, g: torch.Generator) -> torch.Tensor:
    """bf16 [T, Hkv, D] new keys or values: N(0, 1) with max(1, round(0.01 D))
    channels per KV head scaled by 8 (the K/V recipe above), on the CPU."""
    x = torch.randn((T, hkv, d), generator=g, dtype=torch.float32)
    n = max(1, int(round(0.01 * d)))
    for h in range(hkv):
        idx = torch.randperm(d, generator=g)[:n]
        x[:, h, idx] *= 8.0
    return x.to(torch.bfloat16)


@dataclasses.dataclass
class KVWriteWorkload:
    name: str
    key: torch.Tensor                 # bf16 [T, Hkv, D]
    value: torch.Tensor
    slot_mappings: list               # int64 [T] per copy, disjoint slot sets
    num_pages: int                    # pages of the cache all copies write into
    k_descale: float
    v_descale: float
    num_heads_kv: int
    head_dim: int

    @property
    def num_tokens(self) -> int:
        return int(self.key.shape[0])

    def bytes_algorithmic(self) -> int:
        """bf16 read plus E4M3 written, for K and V: 3 bytes per element."""
        return self.num_tokens * self.num_heads_kv * self.head_dim * 2 * 3


KV_WRITE_CONFIG_NAMES = [
    "kv_write_mixed_hd256",  # the 8128 new tokens of the hd256 mixed batch: Hkv 16, D 256
    "kv_write_mixed_hd512",  # the same tokens at D 512, Hkv 4
]


def make_kv_write_config(name: str, device="cpu", copies: int = 1, seed: int = 7) -> KVWriteWorkload:
    """New keys and values of the mixed batch's step: a 4096-token chunk appended
    to a sequence (64 whole pages) and 4032 decode tokens, each the next row of
    its own sequence's last page.  Every copy gets its own pages, so copies never
    share a slot."""
    hkv, d = {"kv_write_mixed_hd256": (16, 256), "kv_write_mixed_hd512": (4, 512)}[name]
    n_chunk, n_dec = 4096, 4032
    T = n_chunk + n_dec
    per_copy = n_chunk // PAGE + n_dec
    pool = copies * per_copy
    g = torch.Generator().manual_seed(seed)
    key = kv_like_values(T, hkv, d, g)
    value = kv_like_values(T, hkv, d, g)
    rng = np.random.default_rng(np.random.PCG64(seed))
    pages = rng.permutation(pool).astype(np.int64)
    maps = []
    for c in range(copies):
        own = pages[c * per_copy:(c + 1) * per_copy]
        chunk = own[: n_chunk // PAGE]
        dec = own[n_chunk // PAGE:]
        sm = np.empty(T, np.int64)
        sm[:n_chunk] = chunk[np.arange(n_chunk) // PAGE] * PAGE + np.arange(n_chunk) % PAGE
        sm[n_chunk:] = dec * PAGE + rng.integers(0, PAGE, size=n_dec)
        maps.append(torch.from_numpy(sm).to(device))
    kd = float(np.float32(np.float32(key.float().abs().amax().item()) / np.float32(448.0)))
    vd = float(np.float32(np.float32(value.float().abs().amax().item()) / np.float32(448.0)))
    return KVWriteWorkload(name=name, key=key.to(device), value=value.to(device), slot_mappings=maps, num_pages=pool,
                           k_descale=kd, v_descale=vd, num_heads_kv=hkv, head_dim=d)


# ------------------------------------------------------------------ LSE-combine inputs

@dataclasses.dataclass
class CombineWorkload:
    name: str
    o_parts: torch.Tensor      # bf16 [P, total_q, Hq, D]
    lse_parts: torch.Tensor    # f32 [P, Hq, total_q]

    def bytes_algorithmic(self) -> int:
        """The parts read (bf16 O and f32 LSE) and the merged row written (bf16 O, f32 LSE)."""
        P, T, hq, d = self.o_parts.shape
        return (P + 1) * T * hq * (2 * d + 4)


COMBINE_CONFIG_NAMES = [
    "lse_combine_mixed_hd512",  # two DCP shards of the hd512 mixed batch's 8128 query rows: Hq 32, D 512
]


def make_combine_config(name: str, device="cpu", seed: int = 11) -> CombineWorkload:
    """Partial outputs N(0, 1) in bf16 and partial LSEs N(0, 3), two parts."""
    P, T, hq, d = {"lse_combine_mixed_hd512": (2, 8128, 32, 512)}[name]
    g = torch.Generator().manual_seed(seed)
    o = torch.randn((P, T, hq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    lse = torch.randn((P, hq, T), generator=g, dtype=torch.float32) * 3.0
    return CombineWorkload(name=name, o_parts=o.to(device), lse_parts=lse.to(device))

