"""CUDA-graph capture of the forward (Q quantization, plan, attention and, when
split, the combine): one capture replays correctly on new input contents.
The split count is a function of host-known sizes only, and the work list is
rebuilt on the device at every replay from the lengths the buffers then hold
(P2 Claims: splits chosen automatically, without the earlier CUDA-graph cap)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import LSE_GATE, TOL, lse_error, oracle_problem, unit_scale_errors

pytestmark = pytest.mark.gpu

CASES = [
    # name, lq, lk, hq, hkv, d, window_left, causal, fp8
    ("decode_hd512_bf16_split", [1] * 7, [1, 64, 129, 700, 1000, 2000, 3000], 32, 4, 512, -1, True, False),
    ("decode_swa_hd256_fp8", [1] * 9, [1, 2, 63, 64, 65, 1024, 1100, 1500, 2000], 32, 16, 256, 1023, True, True),
    ("chunked_hd256_fp8", [37, 100, 1], [300, 300, 5], 8, 4, 256, 100, True, True),
]


def _check(w, out, lse, lk=None):
    ro, rl = oracle.paged_attention(oracle_problem(w, seqused_k=w.lk if lk is None else lk))
    g = out.float().cpu().numpy()
    e = unit_scale_errors(g, ro, w)
    le = lse_error(lse.cpu().numpy(), rl)
    tmax, tmean = TOL[w.fp8_q]
    assert np.isfinite(g).all()
    assert e["max"] <= tmax and e["mean"] <= tmean, (w.name, e, le)
    assert le <= LSE_GATE, (w.name, le)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_captured_forward_replays_on_new_contents(case):
    import fp8_paged_attention_gb300 as fp8pa
    name, lq, lk, hq, hkv, d, wl, causal, fp8 = case
    w1 = synth.make_workload(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=31, device="cuda")
    # same shapes, other values, page permutation and channel scales
    w2 = synth.make_workload(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=32, device="cuda")
    assert w2.k_cache.shape == w1.k_cache.shape and w2.block_table.shape == w1.block_table.shape
    # static buffers hold w1; descales live in device tensors the graph reads
    q, kc, vc = w1.q.clone(), w1.k_cache.clone(), w1.v_cache.clone()
    bt, cu, sk = w1.block_table.clone(), w1.cu_seqlens_q.clone(), w1.seqused_k.clone()
    qd = torch.tensor([w1.q_descale], dtype=torch.float32, device="cuda")
    kd = torch.tensor([w1.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([w1.v_descale], dtype=torch.float32, device="cuda")
    max_lq = int(max(lq))

    def step():
        qq = fp8pa.quantize_q_fp8(q, qd) if fp8 else q
        return fp8pa.fp8_paged_attn_fwd(qq, kc, vc, bt, cu, sk, max_lq, qd, kd, vd, w1.softmax_scale, wl, causal)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()  # warm-up outside the capture (library load, function attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out, lse = step()

    graph.replay()
    torch.cuda.synchronize()
    _check(w1, out, lse)
    out1 = out.clone()

    # New contents in the same buffers: w2's tensors, and shorter contexts for
    # two sequences.  Only sequences whose every key was visible are shortened:
    # pages no query could see hold NaN poison, and a window moved by a shorter
    # context would reach them.
    lk2 = np.asarray(lk, dtype=np.int32).copy()
    first_lo = [max(0, k - q - wl) if wl >= 0 else 0 for q, k in zip(lq, lk)]
    for b in [b for b in range(len(lk)) if first_lo[b] == 0 and lk[b] > 1][-2:]:
        lk2[b] = max(1, lk2[b] - max(1, lk2[b] // 3))
    assert (lk2 != np.asarray(lk)).any()
    q.copy_(w2.q)
    kc.copy_(w2.k_cache)
    vc.copy_(w2.v_cache)
    bt.copy_(w2.block_table)
    sk.copy_(torch.from_numpy(lk2).to("cuda"))
    qd.fill_(w2.q_descale)
    kd.fill_(w2.k_descale)
    vd.fill_(w2.v_descale)
    graph.replay()
    torch.cuda.synchronize()
    _check(w2, out, lse, lk=lk2)
    assert not torch.equal(out, out1)
    assert fp8pa.get_device_status() == 0
