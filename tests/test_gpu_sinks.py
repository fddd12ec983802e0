"""Attention sinks (fp8_paged_attn_fwd_sinks) on every kernel path against the
oracle with the same sinks: decode tiles with and without key splits, E4M3
prefill tiles at head dim 256 and 512, BF16-Q prefill tiles, rows with no
visible key; and sinks at -inf are bit-identical to the call without sinks."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import LSE_GATE, TOL, oracle_problem, unit_scale_errors

pytestmark = pytest.mark.gpu

CASES = {
    # name: (lq, lk, hq, hkv, d, window_left, causal, fp8_q, num_splits)
    "decode_hd256": ([1] * 6, [900, 64, 1500, 3, 700, 2000], 32, 16, 256, 1023, True, True, 1),
    "decode_hd256_split": ([1] * 4, [3000, 2500, 1800, 4000], 32, 16, 256, -1, True, True, 3),
    "decode_hd512_bf16": ([1] * 4, [2100, 900, 64, 1300], 32, 4, 512, -1, True, False, 0),
    "prefill_hd256_fp8": ([200, 65, 1], [600, 65, 300], 32, 16, 256, 255, True, True, 0),
    "prefill_hd512_fp8": ([150, 20], [400, 150], 32, 4, 512, -1, True, True, 0),
    "prefill_hd512_bf16": ([150, 20], [400, 150], 32, 4, 512, -1, True, False, 0),
    "empty_rows": ([3, 2], [1, 0], 4, 2, 256, -1, True, True, 0),
}


def _run(w, sinks, num_splits):
    import fp8_paged_attention_gb300 as fp8pa
    qd = torch.tensor([w.q_descale], dtype=torch.float32, device="cuda")
    kd = torch.tensor([w.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([w.v_descale], dtype=torch.float32, device="cuda")
    q = fp8pa.quantize_q_fp8(w.q, qd) if w.fp8_q else w.q
    return fp8pa.fp8_paged_attn_fwd(q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                                    w.max_seqlen_q, qd, kd, vd, w.softmax_scale, w.window_left, w.causal,
                                    num_splits=num_splits, sinks=sinks)


@pytest.mark.parametrize("name", list(CASES))
def test_sinks_against_oracle(name):
    lq, lk, hq, hkv, d, wl, causal, fp8_q, ns = CASES[name]
    w = synth.make_workload(name, lq, lk, hq, hkv, d, wl, causal, fp8_q, seed=51, device="cuda")
    rng = np.random.default_rng(52)
    sinks = (rng.normal(size=hq) * 3).astype(np.float32)
    sinks[0] = 30.0    # dominates every row of head 0
    sinks[1] = -30.0   # weighs nothing
    out, lse = _run(w, torch.from_numpy(sinks).cuda(), ns)
    ref, ref_lse = oracle.paged_attention(oracle_problem(w, sinks=sinks))
    e = unit_scale_errors(out.float().cpu().numpy(), ref, w)
    tol = TOL[w.fp8_q]
    assert e["max"] <= tol[0] and e["mean"] <= tol[1], e
    g = lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.abs(g[fin] - ref_lse[fin]).max() <= LSE_GATE


@pytest.mark.parametrize("name", ["decode_hd256", "decode_hd256_split", "prefill_hd256_fp8", "prefill_hd512_bf16"])
def test_sinks_at_minus_inf_are_bit_identical_to_no_sinks(name):
    lq, lk, hq, hkv, d, wl, causal, fp8_q, ns = CASES[name]
    w = synth.make_workload(name, lq, lk, hq, hkv, d, wl, causal, fp8_q, seed=53, device="cuda")
    a, la = _run(w, None, ns)
    b, lb = _run(w, torch.full((hq,), -float("inf"), dtype=torch.float32, device="cuda"), ns)
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("name", ["decode_hd256", "decode_hd256_split", "decode_hd512_bf16", "prefill_hd256_fp8",
                                  "prefill_hd512_fp8", "prefill_hd512_bf16"])
def test_null_descales_are_the_unit_scale(name):
    # the no-descale fast path: null q/k/v descales give the bits of descale tensors holding 1.0
    import fp8_paged_attention_gb300 as fp8pa
    lq, lk, hq, hkv, d, wl, causal, fp8_q, ns = CASES[name]
    w = synth.make_workload(name, lq, lk, hq, hkv, d, wl, causal, fp8_q, seed=54, device="cuda")
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    q = fp8pa.quantize_q_fp8(w.q, torch.tensor([w.q_descale], device="cuda")) if fp8_q else w.q
    scale = w.softmax_scale * 0.05  # codes read at unit scale are large: keep the logits moderate
    common = (q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k, w.max_seqlen_q)
    a, la = fp8pa.fp8_paged_attn_fwd(*common, one, one, one, scale, w.window_left, w.causal, num_splits=ns)
    b, lb = fp8pa.fp8_paged_attn_fwd(*common, None, None, None, scale, w.window_left, w.causal, num_splits=ns)
    assert torch.equal(a, b) and torch.equal(la, lb)
    assert torch.isfinite(a.float()).all()
