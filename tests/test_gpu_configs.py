"""Full-size benchmark workloads on the GPU, in the launch configuration the
benchmark times (automatic split count), checked against the oracle on
sampled output rows: a seeded sample of sequences with every query row and
head, plus a sample of the chunked-prefill sequence's rows."""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import LSE_GATE, TOL, lse_error, unit_scale_errors
from tests.test_gpu_attention import run_gpu

pytestmark = pytest.mark.gpu


def sampled_check(w, out, lse, n_seq=12, chunk_tokens=48, seed=0):
    rng = np.random.default_rng(seed)
    B = w.batch
    seqs = sorted(set(rng.choice(B, size=min(n_seq, B), replace=False).tolist()))
    big = [int(b) for b in np.nonzero(w.lq > 64)[0]]
    seqs = sorted(set(seqs) - set(big))
    sub = synth.subproblem_pages(w, seqs + big)
    q = sub["q"]
    if w.fp8_q:
        q = oracle.quantize_q(q, w.q_descale)
    prob = oracle.AttnProblem(q, w.fp8_q, sub["k"], sub["v"], sub["block_table"], sub["cu_seqlens_q"],
                              sub["seqused_k"], w.num_heads_kv, w.q_descale, w.k_descale, w.v_descale,
                              w.softmax_scale, w.window_left, w.causal)
    # rows: every row of the small sequences, a sample of the big ones' tokens
    rows_local, tok_global = [], []
    cu = sub["cu_seqlens_q"]
    toks = sub["tokens"]
    for i, b in enumerate(seqs + big):
        lt = list(range(cu[i], cu[i + 1]))
        if b in big:
            lt = sorted(set(rng.choice(lt, size=min(chunk_tokens, len(lt)), replace=False).tolist())
                        | {lt[0], lt[-1]})
        for t in lt:
            for h in range(w.num_heads_q):
                rows_local.append((t, h))
                tok_global.append((int(toks[t]), h))
    rows_local = np.array(rows_local, dtype=np.int32)
    tok_global = np.array(tok_global, dtype=np.int64)
    ro, rl = oracle.paged_attention(prob, rows=rows_local)
    g = out[torch.from_numpy(tok_global[:, 0]).cuda(), torch.from_numpy(tok_global[:, 1]).cuda()].float().cpu().numpy()
    gl = lse[torch.from_numpy(tok_global[:, 1]).cuda(), torch.from_numpy(tok_global[:, 0]).cuda()].cpu().numpy()
    e = unit_scale_errors(g, ro, w, heads=tok_global[:, 1])
    le = lse_error(gl, rl)
    return e, le, len(rows_local)


@pytest.mark.parametrize("name", ["swa_decode_hd256", "full_decode_hd512_bf16q", "full_decode_hd512_fp8q",
                                  "spec_verify_hd512", "mixed_hd256_swa", "mixed_hd512_causal",
                                  "mixed_hd512_causal_fp8q"])
def test_full_size_config_sampled(name):
    w = synth.make_config(name, device="cuda")
    out, lse = run_gpu(w)
    assert torch.isfinite(out.float()).all()
    e, le, n = sampled_check(w, out, lse)
    print(f"{name}: rows={n} unit-scale max={e['max']:.3e} mean={e['mean']:.3e} raw_max={e['raw_max']:.3e} "
          f"lse_max={le:.3e}")
    tmax, tmean = TOL[w.fp8_q]
    assert e["max"] <= tmax and e["mean"] <= tmean, (name, e, le)
    assert le <= LSE_GATE
    # the same call again gives the same bits
    out2, lse2 = run_gpu(w)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    del w, out, lse, out2, lse2
    gc.collect()
    torch.cuda.empty_cache()
