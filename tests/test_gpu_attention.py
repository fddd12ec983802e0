"""GPU attention vs the fp64 oracle on small and edge-case inputs that span
several 128-key tiles, ragged tails, every row class (decode, verify,
prefill, chunked prefill), windows, empty rows, splits and permuted pages."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import LSE_GATE, TOL, bf16_bits, lse_error, oracle_problem, unit_scale_errors

pytestmark = pytest.mark.gpu


def run_gpu(w, num_splits=0, q8=None, **kw):
    import fp8_paged_attention_gb300 as fp8pa
    dev = w.k_cache.device
    qd = torch.tensor([w.q_descale], dtype=torch.float32, device=dev)
    kd = kw.pop("k_descale", torch.tensor([w.k_descale], dtype=torch.float32, device=dev))
    vd = kw.pop("v_descale", torch.tensor([w.v_descale], dtype=torch.float32, device=dev))
    q = w.q
    if w.fp8_q:
        q = q8 if q8 is not None else fp8pa.quantize_q_fp8(w.q, qd)
    out, lse = fp8pa.fp8_paged_attn_fwd(q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                                        w.max_seqlen_q, qd, kd, vd, w.softmax_scale, w.window_left, w.causal,
                                        num_splits=num_splits, **kw)
    torch.cuda.synchronize()
    return out, lse


def check(w, out, lse, ref=None, prob=None):
    if ref is None:
        ref = oracle.paged_attention(prob if prob is not None else oracle_problem(w))
    ro, rl = ref
    g = out.float().cpu().numpy()
    e = unit_scale_errors(g, ro, w)
    le = lse_error(lse.cpu().numpy(), rl)
    tmax, tmean = TOL[w.fp8_q]
    assert np.isfinite(g).all()
    assert e["max"] <= tmax and e["mean"] <= tmean, (w.name, e, le)
    assert le <= LSE_GATE, (w.name, le)
    return e, le


def make(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=0, **kw):
    return synth.make_workload(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=seed, device="cuda", **kw)


def test_tiny_prefill_config():
    w = synth.make_config("tiny_prefill_hd256", device="cuda")
    out, lse = run_gpu(w)
    check(w, out, lse)


CASES = [
    # name, lq, lk, hq, hkv, d, window_left, causal, fp8
    ("prefill_ragged_hd256", [1, 63, 64, 65, 130, 200], [1, 63, 64, 65, 130, 200], 4, 2, 256, -1, True, True),
    ("prefill_window_hd256", [150, 300], [150, 300], 4, 2, 256, 63, True, True),
    ("chunked_hd256", [37, 100, 1], [300, 300, 5], 8, 4, 256, 100, True, True),
    ("decode_swa_hd256", [1] * 9, [1, 2, 63, 64, 65, 1024, 1100, 1500, 2000], 32, 16, 256, 1023, True, True),
    ("decode_hd512_bf16", [1] * 7, [1, 64, 129, 700, 1000, 2000, 3000], 32, 4, 512, -1, True, False),
    ("decode_hd512_fp8", [1] * 7, [1, 64, 129, 700, 1000, 2000, 3000], 32, 4, 512, -1, True, True),
    ("verify_hd512_bf16", [4] * 5, [4, 65, 300, 1000, 2000], 32, 4, 512, -1, True, False),
    ("verify_hd512_fp8", [4] * 5, [4, 65, 300, 1000, 2000], 32, 4, 512, -1, True, True),
    ("prefill_hd512_bf16", [3, 70, 129], [3, 70, 300], 16, 2, 512, -1, True, False),
    ("prefill_hd512_fp8", [3, 70, 129], [3, 70, 300], 16, 2, 512, -1, True, True),
    ("noncausal_window_hd256", [3, 70], [200, 70], 4, 2, 256, 50, False, True),
    ("noncausal_hd512_bf16", [2, 40], [300, 40], 8, 1, 512, -1, False, False),
    ("mha_group1_hd256", [5, 1], [77, 300], 2, 2, 256, -1, True, True),
    # prefill-class tiles (128 packed rows at hd256): rows and whole sequences with no visible key,
    # one and eight query heads per KV head
    ("prefill_empty_rows_hd256", [20, 12, 30], [10, 0, 30], 4, 2, 256, -1, True, True),
    ("prefill_group1_hd256", [40, 130], [40, 200], 2, 2, 256, -1, True, True),
    ("prefill_group8_window_hd256", [20, 50], [100, 50], 16, 2, 256, 30, True, True),
    ("group16_hd512", [1, 2], [500, 130], 16, 1, 512, -1, True, False),
]


@pytest.mark.parametrize("d,hkv,fp8", [(256, 16, True), (512, 4, True), (512, 4, False)],
                         ids=["hd256_fp8", "hd512_fp8", "hd512_bf16q"])
def test_decode_tiles_never_read_slots_before_the_window(d, hkv, fp8):
    """Decode-shaped tiles read a key union's first page from its first visible
    slot, so the slots before the window may hold anything: here the E4M3 NaN
    code in K and V, which would reach the output through 0 * NaN if they were
    read.  Window starts fall at many offsets within a page; one sequence's
    union lies within one page (that item reads whole pages, so its page is
    left clean).  Auto split and three explicit splits."""
    wl = 700
    lks = [40] + [wl + 2 + 73 * i for i in range(12)]
    w = make(f"trim_{d}_{int(fp8)}", [1] * len(lks), lks, 32, hkv, d, wl, True, fp8, seed=41)
    poisoned = 0
    for b, lk in enumerate(lks):
        lo = max(0, lk - 1 - wl)
        if lo // 64 == (lk - 1) // 64 or lo % 64 == 0:
            continue
        phys = int(w.bt[b, lo // 64])
        w.k_cache[phys, : lo % 64] = 0x7F
        w.v_cache[phys, : lo % 64] = 0x7F
        poisoned += 1
    assert poisoned >= 10
    ref = oracle.paged_attention(oracle_problem(w))
    for splits in (0, 3):
        out, lse = run_gpu(w, num_splits=splits)
        check(w, out, lse, ref=ref)


def test_plan_with_more_long_item_lists_than_its_queue():
    """66 prefill sequences whose item lists are long (6 row tiles x 16 KV
    heads = 96 items each): more than the plan's block-wide queue of 64 holds,
    so the last lists are written by their own warps.  Every row against the
    oracle."""
    w = make("plan_overflow", [321] * 66, [321] * 66, 32, 16, 256, 31, True, True, seed=3)
    out, lse = run_gpu(w)
    check(w, out, lse)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_attention_cases(case):
    name, lq, lk, hq, hkv, d, wl, causal, fp8 = case
    w = make(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=len(name))
    out, lse = run_gpu(w)
    check(w, out, lse)


BF16_CASES = [c for c in CASES if not c[8]]


@pytest.mark.parametrize("case", BF16_CASES, ids=[c[0] for c in BF16_CASES])
def test_bf16_q_literal_v_dequant_path(case):
    """The BF16-Q path with V also dequantized to BF16 (BF16 P, BF16 PV MMA)."""
    import fp8_paged_attention_gb300 as fp8pa
    name, lq, lk, hq, hkv, d, wl, causal, fp8 = case
    w = make(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=len(name) + 1)
    fp8pa.set_bf16_dequant_v(True)
    try:
        out, lse = run_gpu(w)
        out3, lse3 = run_gpu(w, num_splits=3)
    finally:
        fp8pa.set_bf16_dequant_v(False)
    ref = oracle.paged_attention(oracle_problem(w))
    check(w, out, lse, ref=ref)
    check(w, out3, lse3, ref=ref)


def test_empty_rows_and_sequences():
    # seq 0: 5 queries on 3 keys (the first two see nothing); seq 1: no keys; seq 2: no queries
    w = make("empty", [5, 2, 0, 1], [3, 0, 10, 9], 4, 2, 256, -1, True, True)
    out, lse = run_gpu(w)
    ro, rl = oracle.paged_attention(oracle_problem(w))
    g = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for t in (0, 1, 5, 6):
        assert np.all(g[t] == 0) and np.all(l[:, t] == -np.inf)
    check(w, out, lse, ref=(ro, rl))


@pytest.mark.parametrize("fp8", [True, False])
def test_explicit_splits_agree_and_repeat_bit_identically(fp8):
    w = make("splits", [1] * 5 + [4], [3000, 2500, 700, 64, 1, 2000], 32, 4, 512, -1, True, fp8, seed=3)
    ref = oracle.paged_attention(oracle_problem(w))
    for s in (1, 2, 3, 7):
        out, lse = run_gpu(w, num_splits=s)
        check(w, out, lse, ref=ref)
        out2, lse2 = run_gpu(w, num_splits=s)
        assert torch.equal(out, out2) and torch.equal(lse, lse2)


PERM_CASES = [
    # name, lq, lk, hq, hkv, d, window_left, causal, fp8, num_splits, shared_prefix_pages
    ("decode_swa_hd256_e4m3", [1, 1, 3, 40], [900, 1500, 700, 300], 32, 16, 256, 1023, True, True, 0, 0),
    ("prefill_tiles_hd256_e4m3", [200, 1, 150], [400, 900, 150], 8, 4, 256, 100, True, True, 0, 0),
    ("decode_hd512_bf16q", [1] * 5, [90, 700, 1300, 2100, 3000], 32, 4, 512, -1, True, False, 0, 0),
    ("prefill_tiles_hd512_bf16q", [70, 1, 129], [300, 500, 129], 16, 2, 512, -1, True, False, 0, 0),
    ("prefill_tiles_hd512_e4m3", [70, 1, 129], [300, 500, 129], 16, 2, 512, -1, True, True, 0, 0),
    ("decode_hd512_e4m3_split3", [1] * 4, [700, 1300, 2100, 3000], 32, 4, 512, -1, True, True, 3, 0),
    ("decode_hd512_bf16q_split3", [1] * 4, [700, 1300, 2100, 3000], 32, 4, 512, -1, True, False, 3, 0),
    ("verify_shared_prefix_hd512_bf16q", [4] * 6, [1400 + 64 * i for i in range(6)], 32, 4, 512, -1, True, False,
     0, 16),
    ("verify_shared_prefix_hd512_e4m3_split4", [4] * 6, [1400 + 64 * i for i in range(6)], 32, 4, 512, -1, True,
     True, 4, 16),
]


@pytest.mark.parametrize("case", PERM_CASES, ids=[c[0] for c in PERM_CASES])
def test_page_permutation_is_bit_identical(case):
    """Moving the physical pages (cache rows and block table together) changes
    no output bit on any kernel path: decode, prefill tiles of both kernels,
    split KV with the combine, and a prefix whose pages every sequence shares."""
    from tests.helpers import permute_pages
    name, lq, lk, hq, hkv, d, wl, causal, fp8, ns, shared = case
    w = make(name, lq, lk, hq, hkv, d, wl, causal, fp8, seed=11, shared_prefix_pages=shared)
    out1, lse1 = run_gpu(w, num_splits=ns)
    check(w, out1, lse1)
    for seed in (5, 6):
        out2, lse2 = run_gpu(permute_pages(w, seed), num_splits=ns)
        assert torch.equal(out1, out2) and torch.equal(lse1, lse2), (name, seed)


def test_per_batch_head_descales():
    w = make("descale", [1, 2, 1], [500, 300, 900], 8, 2, 256, 200, True, True, seed=9)
    kd = torch.tensor([[w.k_descale, w.k_descale * 0.5], [w.k_descale * 2, w.k_descale],
                       [w.k_descale, w.k_descale * 1.5]], dtype=torch.float32, device="cuda")
    vd = torch.tensor([[w.v_descale, w.v_descale * 2], [w.v_descale * 0.25, w.v_descale],
                       [w.v_descale * 3, w.v_descale]], dtype=torch.float32, device="cuda")
    out, lse = run_gpu(w, k_descale=kd.reshape(-1), v_descale=vd.reshape(-1), descale_batch_stride=2,
                       descale_head_stride=1)
    prob = oracle_problem(w, k_descale=kd.cpu().numpy().ravel(), v_descale=vd.cpu().numpy().ravel(),
                          descale_batch_stride=2, descale_head_stride=1)
    ro, rl = oracle.paged_attention(prob)
    # outputs scale with v_descale: compare on the scale of each sequence's V
    g = out.float().cpu().numpy()
    tok_seq = np.repeat(np.arange(3), w.lq)
    G = 4
    for t in range(w.total_q):
        for h in range(8):
            s = w.v_channel_scale[h // G] * float(vd[tok_seq[t], h // G] / w.v_descale)
            assert np.max(np.abs(g[t, h] - ro[t, h]) / np.maximum(s, np.abs(ro[t, h]))) <= TOL[True][0]
    assert lse_error(lse.cpu().numpy(), rl) <= LSE_GATE


@pytest.mark.parametrize("fp8,limit", [(True, 0), (True, 64), (False, 0)], ids=["e4m3_default_limit",
                                                                                "e4m3_limit64", "bf16_default_limit"])
def test_wait_that_runs_out_sets_timeout_and_context_survives(fp8, limit):
    """A pipeline wait that can never complete (the stall-injection hook) ends on
    its bound: the launch reports DEV_TIMEOUT and the next launch is correct."""
    import fp8_paged_attention_gb300 as fp8pa
    d, hkv = (256, 16) if fp8 else (512, 4)
    w = make("stall", [1] * 5 + [70], [300, 900, 1500, 2000, 64, 200], 32, hkv, d, -1, True, fp8, seed=17)
    fp8pa.reset_device_status()
    fp8pa.set_wait_limit(limit)
    fp8pa.set_stall_injection(True)
    try:
        run_gpu(w)  # synchronizes: the launch ends, without a CUDA error
    finally:
        fp8pa.set_stall_injection(False)
        fp8pa.set_wait_limit(0)
    assert fp8pa.get_device_status() & fp8pa.DEV_TIMEOUT
    fp8pa.reset_device_status()
    out, lse = run_gpu(w)
    check(w, out, lse)
    assert fp8pa.get_device_status() == 0


def test_per_batch_head_descales_prefill_tiles():
    w = make("descale_pf", [40, 70], [200, 70], 8, 2, 256, -1, True, True, seed=13)
    kd = torch.tensor([[w.k_descale, w.k_descale * 0.5], [w.k_descale * 2, w.k_descale]], dtype=torch.float32,
                      device="cuda")
    vd = torch.tensor([[w.v_descale * 3, w.v_descale], [w.v_descale, w.v_descale * 0.25]], dtype=torch.float32,
                      device="cuda")
    out, lse = run_gpu(w, k_descale=kd.reshape(-1), v_descale=vd.reshape(-1), descale_batch_stride=2,
                       descale_head_stride=1)
    prob = oracle_problem(w, k_descale=kd.cpu().numpy().ravel(), v_descale=vd.cpu().numpy().ravel(),
                          descale_batch_stride=2, descale_head_stride=1)
    ro, rl = oracle.paged_attention(prob)
    g = out.float().cpu().numpy()
    tok_seq = np.repeat(np.arange(2), w.lq)
    G = 4
    for t in range(w.total_q):
        for h in range(8):
            s = w.v_channel_scale[h // G] * float(vd[tok_seq[t], h // G] / w.v_descale)
            assert np.max(np.abs(g[t, h] - ro[t, h]) / np.maximum(s, np.abs(ro[t, h]))) <= TOL[True][0]
    assert lse_error(lse.cpu().numpy(), rl) <= LSE_GATE


@pytest.mark.parametrize("d,sharp", [(256, 8.0), (256, 0.1), (512, 8.0), (512, 0.1)],
                         ids=["hd256_sharp", "hd256_flat", "hd512_sharp", "hd512_flat"])
def test_prefill_tiles_sharp_and_flat_softmax(d, sharp):
    """Prefill tiles under a sharp softmax (scores scaled by 8: a few keys carry
    each row's mass, where P's E4M3 rounding matters most) and a flat one
    (scaled by 0.1: every weight small).  Both match the oracle."""
    hq = 8 if d == 256 else 16
    w = make("sharp", [70, 130], [300, 130], hq, 2, d, -1, True, True, seed=41)
    w = synth.Workload(**{**w.__dict__, "softmax_scale": w.softmax_scale * sharp})
    out, lse = run_gpu(w)
    check(w, out, lse)


def test_bad_page_id_in_prefill_tiles_sets_status():
    import fp8_paged_attention_gb300 as fp8pa
    w = make("badpage_pf", [40, 50], [200, 300], 4, 2, 256, -1, True, True, seed=6)
    bt = w.block_table.clone()
    bt[1, 1] = 1 << 20
    fp8pa.reset_device_status()
    out, lse = run_gpu(synth.Workload(**{**w.__dict__, "block_table": bt}))
    assert fp8pa.get_device_status() & fp8pa.DEV_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    # sequence 0 does not reference the bad entry
    ro, rl = oracle.paged_attention(oracle_problem(w))
    e = unit_scale_errors(out.float().cpu().numpy()[:40], ro[:40], w)
    assert e["max"] <= TOL[True][0]
    fp8pa.reset_device_status()


def test_bad_page_id_sets_status_and_reads_zeros():
    import fp8_paged_attention_gb300 as fp8pa
    w = make("badpage", [1, 1], [200, 300], 8, 4, 256, -1, True, True, seed=4)
    bt = w.block_table.clone()
    bt[1, 2] = 1 << 20
    fp8pa.reset_device_status()
    out, lse = run_gpu(synth.Workload(**{**w.__dict__, "block_table": bt}))
    st = fp8pa.get_device_status()
    assert st & fp8pa.DEV_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    # sequence 0 is untouched by the bad entry
    ro, rl = oracle.paged_attention(oracle_problem(w))
    e = unit_scale_errors(out.float().cpu().numpy()[:1], ro[:1], w)
    assert e["max"] <= TOL[True][0]
    fp8pa.reset_device_status()
    assert fp8pa.get_device_status() == 0


@pytest.mark.parametrize("lq,literal_v", [(16, False), (1, False), (16, True)],
                         ids=["prefill_tiles", "decode_tile", "prefill_tiles_literal_v"])
def test_bf16_q_path_dequantizes_every_k_code_exactly(lq, literal_v):
    """BF16-Q path: a single visible key whose 512 channels hold every finite
    E4M3 code, and one-hot query rows of several magnitudes (1, 2^-30, 2^20, 3).
    With one key the lse is the score itself, softmax_scale * q * dec(code), so
    a code decoded wrongly (a flushed subnormal, a wrong exponent) or a Q row
    scaled wrongly shows at f32 precision."""
    import fp8_paged_attention_gb300 as fp8pa
    hq, d = 16, 512
    codes = np.arange(d) % 256
    codes[codes == 0x7F] = 0x00
    codes[codes == 0xFF] = 0x80
    kc = torch.zeros((2, 64, 1, d), dtype=torch.uint8)
    vc = torch.zeros((2, 64, 1, d), dtype=torch.uint8)
    kc[0, 0, 0] = torch.from_numpy(codes.astype(np.uint8))
    vc[0, 0, 0] = 0x38  # 1.0
    qvals = [1.0, 2.0 ** -30, 2.0 ** 20, 3.0]
    rows = lq * hq
    q = torch.zeros((lq, hq, d), dtype=torch.float32)
    want = np.zeros((hq, lq))
    dec = oracle.e4m3_decode(codes)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    for r in range(rows):
        t, h = divmod(r, hq)
        ch = (r * 37) % 256 if rows < 256 else r % 256
        qv = qvals[r % len(qvals)]
        q[t, h, ch] = qv
        want[h, t] = scale * qv * dec[ch]
    q = q.to(torch.bfloat16).cuda()
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    fp8pa.set_bf16_dequant_v(literal_v)
    try:
        out, lse = fp8pa.fp8_paged_attn_fwd(q, kc.cuda(), vc.cuda(), torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                                            torch.tensor([0, lq], dtype=torch.int32, device="cuda"),
                                            torch.tensor([1], dtype=torch.int32, device="cuda"), lq, one, one, one,
                                            scale, -1, False)
        torch.cuda.synchronize()
    finally:
        fp8pa.set_bf16_dequant_v(False)
    got = lse.cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    assert np.all(err <= 2e-6 + 1e-5 * np.abs(want)), (err.max(), np.unravel_index(err.argmax(), err.shape))
    assert torch.equal(out.float().cpu(), torch.ones((lq, hq, d)))  # the one V row, all 1.0


@pytest.mark.parametrize("lq", [16, 1])
def test_bf16_q_split_carries_full_mantissa_rows(lq):
    """BF16-Q path: with one visible key the lse is the score itself, so it shows
    how exactly the kernel carries Q.  Rows of full-mantissa BF16 values: N(0, 1)
    rows, rows whose values all lie within [2^-9, 1] of the row's largest, and
    rows spanning 2^-30 .. 2^20 in magnitude.  The kernel's E4M3 pair holds every
    value down to 2^-9 of the row's largest exactly, so those terms must agree
    with fp64 to f32 accumulation accuracy; a smaller value is off by at most
    its own magnitude, which the bound allows for."""
    import fp8_paged_attention_gb300 as fp8pa
    hq, d = 16, 512
    rng = np.random.default_rng(77)
    codes = rng.integers(0, 256, size=d)
    codes[(codes & 0x7F) == 0x7F] = 0x38
    kc = torch.zeros((2, 64, 1, d), dtype=torch.uint8)
    vc = torch.zeros((2, 64, 1, d), dtype=torch.uint8)
    kc[0, 0, 0] = torch.from_numpy(codes.astype(np.uint8))
    vc[0, 0, 0] = 0x38  # 1.0
    dec = oracle.e4m3_decode(codes).astype(np.float64)
    q = np.zeros((lq, hq, d), dtype=np.float32)
    for t in range(lq):
        for h in range(hq):
            kind = (t * hq + h) % 3
            if kind == 0:
                row = rng.standard_normal(d)
            elif kind == 1:
                row = rng.choice([-1.0, 1.0], d) * np.exp2(rng.uniform(-9.0, 0.0, d))
            else:
                row = rng.choice([-1.0, 1.0], d) * np.exp2(rng.uniform(-30.0, 20.0, d))
            q[t, h] = row
    qb = torch.from_numpy(q).to(torch.bfloat16)
    qv = qb.float().numpy().astype(np.float64)  # the BF16 values the kernel sees
    scale = float(np.float32(1.0 / np.sqrt(d)))
    want = scale * np.einsum("thd,d->ht", qv, dec)
    bound = scale * np.einsum("thd,d->ht", np.abs(qv), np.abs(dec))
    small = np.abs(qv) < np.exp2(-9.0) * np.abs(qv).max(axis=2, keepdims=True)
    slack = scale * np.einsum("thd,d->ht", np.abs(qv) * small, np.abs(dec))
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    out, lse = fp8pa.fp8_paged_attn_fwd(qb.cuda(), kc.cuda(), vc.cuda(), torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                                        torch.tensor([0, lq], dtype=torch.int32, device="cuda"),
                                        torch.tensor([1], dtype=torch.int32, device="cuda"), lq, one, one, one,
                                        scale, -1, False)
    torch.cuda.synchronize()
    got = lse.cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    assert np.all(err <= 2e-6 * bound + slack + 1e-30), (float((err / np.maximum(bound, 1e-30)).max()),)
    exact_rows = ~small.any(axis=2).T  # rows with no value below 2^-9 of their largest
    assert exact_rows.any() and np.all(err[exact_rows] <= 2e-6 * bound[exact_rows])
    assert torch.equal(out.float().cpu(), torch.ones((lq, hq, d)))
