"""fp8_paged_attn_fwd_noalloc — the forward for callers that cannot allocate
device memory at call time (an engine that pre-reserves nearly all HBM for its
KV-cache pool, a plugin host without an allocator).  It keeps its scratch in a
fixed device array inside the library.  These tests call it through the C ABI
and check that, on two calls in a row, it gives what the workspace entry
point gives: the same kernels run with the same split count, so the outputs
agree bit for bit (which also puts them within the tolerances the other GPU
tests use).  They also check that it refuses a call whose scratch need
exceeds the array.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests.helpers import LSE_GATE, TOL, lse_error, unit_scale_errors

pytestmark = pytest.mark.gpu

CASES = [
    # name, lq, lk, hq, hkv, d, window_left, causal, fp8_q, num_splits
    ("decode_hd256_fp8", [1] * 6, [90, 700, 1100, 1500, 2000, 64], 32, 16, 256, 1023, True, True, 0),
    ("decode_hd512_bf16_split3", [1] * 4, [300, 1000, 2000, 3000], 32, 4, 512, -1, True, False, 3),
    ("verify_hd512_fp8_split5", [4] * 3, [200, 1300, 2500], 32, 4, 512, -1, True, True, 5),
    ("prefill_hd256_fp8", [70, 1, 130], [70, 500, 300], 8, 4, 256, 100, True, True, 0),
]


def _args(w, q, qd, kd, vd, num_splits, out, lse):
    import fp8_paged_attention_gb300 as fp8pa
    stream = torch.cuda.current_stream().cuda_stream
    return [q.data_ptr(), fp8pa.FP8PA_E4M3 if w.fp8_q else fp8pa.FP8PA_BF16, w.k_cache.data_ptr(),
            w.v_cache.data_ptr(), w.num_pages, w.block_table.data_ptr(), w.block_table.shape[1],
            w.cu_seqlens_q.data_ptr(), w.seqused_k.data_ptr(), w.batch, w.total_q, w.max_seqlen_q, w.num_heads_q,
            w.num_heads_kv, w.head_dim, qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), 0, 0,
            ctypes.c_float(w.softmax_scale), w.window_left, int(w.causal), num_splits, out.data_ptr(),
            lse.data_ptr(), stream]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point(case):
    import fp8_paged_attention_gb300 as fp8pa
    name, lq, lk, hq, hkv, d, wl, causal, fp8, ns = case
    w = synth.make_workload(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=21, device="cuda")
    qd = torch.tensor([w.q_descale], dtype=torch.float32, device="cuda")
    kd = torch.tensor([w.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([w.v_descale], dtype=torch.float32, device="cuda")
    q = fp8pa.quantize_q_fp8(w.q, qd) if fp8 else w.q
    ref_out, ref_lse = fp8pa.fp8_paged_attn_fwd(q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                                                w.seqused_k, w.max_seqlen_q, qd, kd, vd, w.softmax_scale, wl,
                                                causal, num_splits=ns)
    torch.cuda.synchronize()
    lib = fp8pa.load_library()
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    for _call in range(2):
        # the second call starts from whatever the first left in the shared scratch
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        rc = lib.fp8_paged_attn_fwd_noalloc(*_args(w, q, qd, kd, vd, ns, out, lse))
        assert rc == 0, lib.fp8pa_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), (name, _call)
        e = unit_scale_errors(out.float().cpu().numpy(), ref_out.float().cpu().numpy().astype(np.float64), w)
        le = lse_error(lse.cpu().numpy(), ref_lse.cpu().numpy().astype(np.float64))
        tmax, tmean = TOL[fp8]
        assert e["max"] <= tmax and e["mean"] <= tmean, (name, e)
        assert le <= LSE_GATE, (name, le)


def test_noalloc_automatic_splits_step_down_to_fit_its_scratch():
    # 64 sequences x 4 verify tokens, Hq 32 / Hkv 4, D 512: the automatic rule picks 4 splits for these
    # 32-row tiles, whose partials need more than the scratch holds; the call runs the largest split
    # count that fits and gives exactly what the workspace entry point gives with that count
    import fp8_paged_attention_gb300 as fp8pa
    lk = [2048 + 13 * i for i in range(64)]
    w = synth.make_workload("verify_steps_down", [4] * 64, lk, 32, 4, 512, -1, True, False, seed=7, device="cuda")
    mp = w.block_table.shape[1]
    s_auto = fp8pa.num_splits(w.batch, w.total_q, w.max_seqlen_q, 32, 4, 512, fp8pa.FP8PA_BF16, mp, -1, 0)
    assert s_auto > 1
    assert fp8pa.workspace_size(w.batch, w.total_q, w.max_seqlen_q, 32, 4, 512, fp8pa.FP8PA_BF16, mp, -1, 0) > (32 << 20)
    fits = [s for s in range(1, s_auto) if fp8pa.workspace_size(w.batch, w.total_q, w.max_seqlen_q, 32, 4, 512,
                                                                 fp8pa.FP8PA_BF16, mp, -1, s) <= (32 << 20)]
    s_fit = max(fits)
    qd = torch.ones(1, dtype=torch.float32, device="cuda")
    kd = torch.tensor([w.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([w.v_descale], dtype=torch.float32, device="cuda")
    ref_out, ref_lse = fp8pa.fp8_paged_attn_fwd(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                                                w.max_seqlen_q, qd, kd, vd, w.softmax_scale, -1, True,
                                                num_splits=s_fit)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    lib = fp8pa.load_library()
    rc = lib.fp8_paged_attn_fwd_noalloc(*_args(w, w.q, qd, kd, vd, 0, out, lse))
    assert rc == 0, lib.fp8pa_last_error().decode()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_calls_beyond_its_scratch():
    import fp8_paged_attention_gb300 as fp8pa
    w = synth.make_workload("big_split", [1] * 64, [4096] * 64, 32, 4, 512, -1, True, False, seed=5, device="cuda")
    ns = 64
    need = fp8pa.workspace_size(w.batch, w.total_q, w.max_seqlen_q, 32, 4, 512, fp8pa.FP8PA_BF16,
                                w.block_table.shape[1], -1, ns)
    assert need > (32 << 20)
    qd = torch.ones(1, dtype=torch.float32, device="cuda")
    out = torch.full((w.total_q, 32, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((32, w.total_q), 7.0, dtype=torch.float32, device="cuda")
    lib = fp8pa.load_library()
    rc = lib.fp8_paged_attn_fwd_noalloc(*_args(w, w.q, qd, qd, qd, ns, out, lse))
    assert rc == fp8pa.Fp8paError(1, "").status == 1
    msg = lib.fp8pa_last_error().decode()
    assert "scratch" in msg and str(need) in msg
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())  # nothing was launched
