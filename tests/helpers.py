"""Shared test helpers: build oracle problems from synthetic workloads or from
hand-made page contents."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

PAGE = 64


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_problem(w: synth.Workload, q_codes: np.ndarray | None = None, **over) -> oracle.AttnProblem:
    """Oracle view of a synthetic workload.  On the FP8 path Q is the oracle's
    own E4M3 quantization of the bf16 Q (unless q_codes is given)."""
    qb = bf16_bits(w.q)
    if w.fp8_q:
        q = q_codes if q_codes is not None else oracle.quantize_q(qb, w.q_descale)
    else:
        q = qb
    kw = dict(q=q, q_is_e4m3=w.fp8_q, k_cache=w.k_cache.cpu().numpy(), v_cache=w.v_cache.cpu().numpy(),
              block_table=w.bt, cu_seqlens_q=w.cu_seqlens_q.cpu().numpy(), seqused_k=w.lk,
              num_heads_kv=w.num_heads_kv, q_descale=w.q_descale, k_descale=w.k_descale,
              v_descale=w.v_descale, softmax_scale=w.softmax_scale, window_left=w.window_left,
              causal=w.causal)
    kw.update(over)
    return oracle.AttnProblem(**kw)


def paged_from_logical(k_logical, v_logical, lk, rng, poison=0x7F, extra_pages=0):
    """Lay per-sequence logical K/V rows ([Lk, Hkv, D] uint8 each) into a
    randomly permuted paged cache.  Returns (k_cache, v_cache, block_table)."""
    B = len(lk)
    pages = [(int(n) + PAGE - 1) // PAGE for n in lk]
    n_phys = sum(pages) + 1 + extra_pages
    hkv, d = k_logical[0].shape[1], k_logical[0].shape[2]
    perm = rng.permutation(n_phys)
    kc = np.full((n_phys, PAGE, hkv, d), poison, dtype=np.uint8)
    vc = np.full((n_phys, PAGE, hkv, d), poison, dtype=np.uint8)
    bt = np.full((B, max(1, max(pages) if pages else 1)), perm[-1], dtype=np.int32)
    nxt = 0
    for b in range(B):
        for j in range(pages[b]):
            phys = int(perm[nxt])
            nxt += 1
            bt[b, j] = phys
            s0, s1 = j * PAGE, min(int(lk[b]), (j + 1) * PAGE)
            kc[phys, : s1 - s0] = k_logical[b][s0:s1]
            vc[phys, : s1 - s0] = v_logical[b][s0:s1]
    return kc, vc, bt


def cu_from_lq(lq):
    cu = np.zeros((len(lq) + 1,), dtype=np.int32)
    cu[1:] = np.cumsum(lq)
    return cu


# Tolerances on unit-scale outputs: (max, mean) of |gpu - oracle| / max(s, |oracle|),
# where s is the scale the V channel was drawn with (1, or 8 for the boosted
# channels).  The output is bf16, which carries up to 2^-9 of |o| of rounding
# error whatever the arithmetic, so an output above its channel's scale is
# measured relative to its own magnitude.
TOL = {True: (3e-2, 3e-3), False: (1e-2, 1e-3)}   # keyed by "FP8-MMA path"
LSE_REPORT = {True: 2e-2, False: 5e-3}            # reported; gated only loosely
LSE_GATE = 0.1


def unit_scale_errors(gpu_out: np.ndarray, ref_out: np.ndarray, w, heads=None):
    """gpu_out, ref_out: [rows, Hq, D] (or [rows, D] with heads giving each row's head)."""
    G = w.num_heads_q // w.num_heads_kv
    if heads is None:
        s = w.v_channel_scale[np.arange(w.num_heads_q) // G][None, :, :]
    else:
        s = w.v_channel_scale[np.asarray(heads) // G]
    diff = np.abs(gpu_out.astype(np.float64) - ref_out)
    e = diff / np.maximum(s, np.abs(ref_out))
    return dict(max=float(e.max()) if e.size else 0.0, mean=float(e.mean()) if e.size else 0.0,
                raw_max=float(diff.max()) if diff.size else 0.0)


def lse_error(gpu_lse: np.ndarray, ref_lse: np.ndarray):
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(gpu_lse), fin), "empty rows must give lse = -inf exactly"
    assert np.all(gpu_lse[~fin] == -np.inf)
    return float(np.abs(gpu_lse[fin] - ref_lse[fin]).max()) if fin.any() else 0.0


def permute_pages(w: synth.Workload, seed: int) -> synth.Workload:
    """The same workload with its physical pages moved by a random permutation
    (cache rows and block-table entries together).  Pages shared by several
    sequences stay shared; every logical page keeps its contents."""
    n = w.num_pages
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(seed)).to(w.k_cache.device)
    kc = torch.empty_like(w.k_cache)
    vc = torch.empty_like(w.v_cache)
    kc[perm] = w.k_cache
    vc[perm] = w.v_cache
    bt = perm.to(torch.int32)[w.block_table.long()].contiguous()
    bt_host = bt.cpu().numpy()
    return synth.Workload(**{**w.__dict__, "k_cache": kc, "v_cache": vc, "block_table": bt, "bt": bt_host,
                             "poison_page": int(perm[w.poison_page])})
