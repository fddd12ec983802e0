"""The context call of decode-context parallelism (DCP): attention of the
query tokens over shards of the context keys, each shard's non-causal call run
as local attention with a window covering every key, and the partials merged by
fp8pa_lse_combine.  Checked against the oracle's attention over all keys, and
the combine on its own against the oracle's combine."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import LSE_GATE, TOL, bf16_bits, oracle_problem, unit_scale_errors

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("parts", [1, 2, 3, 5])
def test_lse_combine_matches_oracle(parts):
    import fp8_paged_attention_gb300 as fp8pa
    rng = np.random.default_rng(parts)
    T, hq, d = 37, 8, 512
    o = torch.from_numpy(rng.normal(size=(parts, T, hq, d)).astype(np.float32)).to(torch.bfloat16)
    lse = (rng.normal(size=(parts, hq, T)) * 3).astype(np.float32)
    lse[rng.random(size=lse.shape) < 0.2] = -np.inf   # empty shards
    lse[:, 1, 4] = -np.inf                            # a row no shard sees
    got, got_lse = fp8pa.lse_combine(o.cuda(), torch.from_numpy(lse).cuda())
    want, want_lse = oracle.lse_combine(bf16_bits(o), lse)
    g = got.float().cpu().numpy()
    err = np.abs(g - want) / np.maximum(1.0, np.abs(want))
    assert err.max() <= 4e-3, err.max()
    gl = got_lse.cpu().numpy()
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(gl), fin) and np.all(gl[~fin] == -np.inf)
    assert np.all(g[~fin.T] == 0)  # rows no shard sees: out = 0
    assert np.abs(gl[fin] - want_lse[fin]).max() <= 1e-5 * max(1.0, np.abs(want_lse[fin]).max())


def _shard_calls(w, cuts, window_left, q, qd, kd, vd):
    """Forward over each shard of every sequence's context pages; returns stacked (out, lse)."""
    import fp8_paged_attention_gb300 as fp8pa
    outs, lses = [], []
    bounds = [0] + list(cuts) + [None]
    for p0, p1 in zip(bounds[:-1], bounds[1:]):
        n = []
        pages = []
        for b in range(w.batch):
            lk = int(w.lk[b])
            lo = p0 * 64
            hi = lk if p1 is None else min(lk, p1 * 64)
            n.append(max(0, hi - lo))
            pages.append(w.bt[b, p0:(w.bt.shape[1] if p1 is None else p1)])
        width = max(1, max(len(x) for x in pages))
        bt = np.full((w.batch, width), w.poison_page, np.int32)
        for b, x in enumerate(pages):
            bt[b, :len(x)] = x
        out, lse = fp8pa.fp8_paged_attn_fwd(q, w.k_cache, w.v_cache, torch.from_numpy(bt).cuda(), w.cu_seqlens_q,
                                            torch.tensor(n, dtype=torch.int32).cuda(), w.max_seqlen_q, qd, kd, vd,
                                            w.softmax_scale, window_left, False)
        outs.append(out)
        lses.append(lse)
    return torch.stack(outs), torch.stack(lses)


@pytest.mark.parametrize("hd,fp8_q", [(512, False), (512, True), (256, True)])
def test_dcp_context_shards_combine_to_the_whole_context(hd, fp8_q):
    import fp8_paged_attention_gb300 as fp8pa
    hq, hkv = (32, 4) if hd == 512 else (32, 16)
    lq = [16, 5, 1, 9]
    lk = [700, 1000, 333, 512]
    w = synth.make_workload(f"dcp_{hd}", lq, lk, hq, hkv, hd, -1, False, fp8_q, seed=31, device="cuda")
    qd = torch.tensor([w.q_descale], dtype=torch.float32, device="cuda")
    kd = torch.tensor([w.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([w.v_descale], dtype=torch.float32, device="cuda")
    q = fp8pa.quantize_q_fp8(w.q, qd) if fp8_q else w.q
    full_cover = int(max(lk))
    # the context call as local attention with a window covering every key: the same mask as non-causal
    a, la = fp8pa.fp8_paged_attn_fwd(q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                                     w.max_seqlen_q, qd, kd, vd, w.softmax_scale, -1, False)
    b, lb = fp8pa.fp8_paged_attn_fwd(q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                                     w.max_seqlen_q, qd, kd, vd, w.softmax_scale, full_cover, False)
    assert torch.equal(a, b) and torch.equal(la, lb)
    # two and three context shards (page boundaries), combined by their LSE
    ref, ref_lse = oracle.paged_attention(oracle_problem(w))
    for cuts in ([5], [3, 9]):
        parts, lses = _shard_calls(w, cuts, full_cover, q, qd, kd, vd)
        out, lse = fp8pa.lse_combine(parts.contiguous(), lses.contiguous())
        e = unit_scale_errors(out.float().cpu().numpy(), ref, w)
        tol = TOL[fp8_q]
        assert e["max"] <= tol[0] and e["mean"] <= tol[1], (cuts, e)
        fin = np.isfinite(ref_lse)
        assert np.abs(lse.cpu().numpy()[fin] - ref_lse[fin]).max() <= LSE_GATE
