"""fp8pa_kv_cache_write on the GPU against the oracle: the whole cache is
bit-identical (written slots and the poison around them), for both head-dim
layouts, ragged token counts, padding slots, strided token rows, special values
and slots past the cache."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(seed, T, hkv, d, pool_pages, pad_frac=0.1):
    g = torch.Generator().manual_seed(seed)
    k = synth.kv_like_values(T, hkv, d, g)
    v = synth.kv_like_values(T, hkv, d, g)
    rng = np.random.default_rng(seed)
    slots = rng.permutation(pool_pages * 64)[:T].astype(np.int64)
    slots[rng.random(T) < pad_frac] = -1
    kd = float(k.abs().max()) / 448.0
    vd = float(v.abs().max()) / 448.0
    return k, v, slots, kd, vd


def _run_both(k, v, slots, kd, vd, pool_pages, key_view=None, value_view=None):
    import fp8_paged_attention_gb300 as fp8pa
    T, hkv, d = k.shape
    kc = torch.full((pool_pages, 64, hkv, d), 0x7F, dtype=torch.uint8, device="cuda")
    vc = torch.full_like(kc, 0x7F)
    kdt = torch.tensor([kd], dtype=torch.float32, device="cuda")
    vdt = torch.tensor([vd], dtype=torch.float32, device="cuda")
    fp8pa.kv_cache_write(k.cuda() if key_view is None else key_view, v.cuda() if value_view is None else value_view,
                         kc, vc, torch.from_numpy(slots).cuda(), kdt, vdt)
    okc = np.full((pool_pages, 64, hkv, d), 0x7F, np.uint8)
    ovc = np.full_like(okc, 0x7F)
    bad = oracle.kv_cache_write(_bits(k), _bits(v), slots, float(np.float32(kd)), float(np.float32(vd)), okc, ovc)
    return kc.cpu().numpy(), vc.cpu().numpy(), okc, ovc, bad


@pytest.mark.parametrize("hkv,d,T", [(16, 256, 517), (4, 512, 333), (16, 256, 1), (2, 64, 70), (3, 512, 97),
                                     (5, 200, 45), (6, 512, 1000)])
def test_kv_write_bit_exact_against_oracle(hkv, d, T):
    pool = (T + 63) // 64 * 2 + 1
    k, v, slots, kd, vd = _case(T * 7 + d, T, hkv, d, pool)
    kc, vc, okc, ovc, bad = _run_both(k, v, slots, kd, vd, pool)
    assert bad == 0
    assert np.array_equal(kc, okc), np.argwhere(kc != okc)[:5]
    assert np.array_equal(vc, ovc), np.argwhere(vc != ovc)[:5]


def test_kv_write_strided_rows_of_a_fused_buffer():
    T, hkv, d, pool = 200, 4, 512, 8
    k, v, slots, kd, vd = _case(11, T, hkv, d, pool)
    fused = torch.empty((T, 3, hkv, d), dtype=torch.bfloat16, device="cuda")
    fused[:, 1] = k.cuda()
    fused[:, 2] = v.cuda()
    kc, vc, okc, ovc, _ = _run_both(k, v, slots, kd, vd, pool, key_view=fused[:, 1], value_view=fused[:, 2])
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)


def test_kv_write_special_values_bit_exact():
    T, hkv, d, pool = 64, 2, 64, 2
    vals = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e30, -1e30, 1e-30, 448.0, 464.0, 465.0, -3.0],
                    dtype=np.float32)
    rng = np.random.default_rng(12)
    k = torch.from_numpy(rng.choice(vals, size=(T, hkv, d))).to(torch.bfloat16)
    v = torch.from_numpy(rng.choice(vals, size=(T, hkv, d)) * 0.5).to(torch.bfloat16)
    slots = rng.permutation(pool * 64)[:T].astype(np.int64)
    kc, vc, okc, ovc, _ = _run_both(k, v, slots, 1.0, 0.37, pool)
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)


def test_kv_write_slot_past_cache_sets_status_and_skips():
    import fp8_paged_attention_gb300 as fp8pa
    T, hkv, d, pool = 30, 2, 64, 1
    k, v, slots, kd, vd = _case(13, T, hkv, d, pool, pad_frac=0.0)
    slots[3] = pool * 64 + 5
    slots[17] = 10 ** 9
    fp8pa.reset_device_status()
    torch.cuda.synchronize()
    kc, vc, okc, ovc, bad = _run_both(k, v, slots, kd, vd, pool)
    assert bad == 2
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)
    st = fp8pa.get_device_status()
    assert st & fp8pa.DEV_BAD_SLOT
    fp8pa.reset_device_status()


def test_kv_write_then_attention_reads_what_was_written():
    # one sequence written through the slot mapping, then read by the forward:
    # the same output as the oracle's attention over the oracle-written cache
    import fp8_paged_attention_gb300 as fp8pa
    from tests.helpers import TOL, unit_scale_errors
    Lk, hkv, G, d, pool = 300, 4, 8, 512, 12
    k, v, _, kd, vd = _case(14, Lk, hkv, d, pool, pad_frac=0.0)
    rng = np.random.default_rng(14)
    n_pages = (Lk + 63) // 64
    phys = rng.permutation(pool)[:n_pages]
    slots = np.array([phys[t // 64] * 64 + t % 64 for t in range(Lk)], np.int64)
    kc, vc, okc, ovc, _ = _run_both(k, v, slots, kd, vd, pool)
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)
    bt = torch.tensor(phys[None, :], dtype=torch.int32)
    q = (torch.randn((4, hkv * G, d), generator=torch.Generator().manual_seed(15))).to(torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    su = torch.tensor([Lk], dtype=torch.int32)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    out, _ = fp8pa.fp8_paged_attn_fwd(q.cuda(), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(), bt.cuda(),
                                      cu.cuda(), su.cuda(), 4, one, torch.tensor([kd], device="cuda"),
                                      torch.tensor([vd], device="cuda"), d ** -0.5, -1, True)
    prob = oracle.AttnProblem(q=_bits(q), q_is_e4m3=False, k_cache=okc, v_cache=ovc, block_table=bt.numpy(),
                              cu_seqlens_q=cu.numpy(), seqused_k=su.numpy(), num_heads_kv=hkv, q_descale=1.0,
                              k_descale=float(np.float32(kd)), v_descale=float(np.float32(vd)),
                              softmax_scale=d ** -0.5, window_left=-1, causal=True)
    want, _ = oracle.paged_attention(prob)
    o = out.float().cpu().numpy()
    err = np.abs(o - want) / np.maximum(1.0, np.abs(want))
    assert err.max() <= TOL[False][0] and err.mean() <= TOL[False][1], (err.max(), err.mean())


@pytest.mark.parametrize("kd,vd", [(5 / 64, 3 / 64), (0.75, 5.0), (35 / 448, 1.0)],
                         ids=["short_mantissa_5_64_3_64", "short_mantissa_0.75_5", "short_35_448_and_unit"])
def test_kv_write_every_bf16_pattern_with_short_mantissa_descales(kd, vd):
    """Every bf16 bit pattern as a key and a value, under descales whose short
    mantissas put many quotients exactly on E4M3 rounding boundaries, where the
    division-free quotient must round exactly as the IEEE division does.  The
    cache matches the oracle bit for bit."""
    T, hkv, d, pool = 128, 2, 256, 3
    pat = np.arange(65536, dtype=np.uint16)
    rng = np.random.default_rng(31)
    k = torch.from_numpy(rng.permutation(pat).astype(np.int16).reshape(T, hkv, d)).view(torch.bfloat16)
    v = torch.from_numpy(rng.permutation(pat).astype(np.int16).reshape(T, hkv, d)).view(torch.bfloat16)
    slots = rng.permutation(pool * 64)[:T].astype(np.int64)
    kc, vc, okc, ovc, bad = _run_both(k, v, slots, kd, vd, pool)
    assert bad == 0
    assert np.array_equal(kc, okc), np.argwhere(kc != okc)[:5]
    assert np.array_equal(vc, ovc), np.argwhere(vc != ovc)[:5]


def _fast_range_descales():
    """fp32 descales across the division-free quantizer's range [2^-64, 2^64],
    its two edges and the values just outside them (those take the division),
    mantissas of all ones, and mantissas 2^20 a +- s, which put quotients of
    bf16 inputs very close to fp32 rounding midpoints next to E4M3 boundaries."""
    rng = np.random.default_rng(2024)
    ds = [2.0 ** -64, 2.0 ** 64, float(np.nextafter(np.float32(2.0 ** -64), np.float32(0))),
          float(np.nextafter(np.float32(2.0 ** 64), np.float32(np.inf)))]
    ds += list(2.0 ** rng.uniform(-64, 64, 12)) + list(10.0 ** rng.uniform(-4, 2, 8))
    ds += [np.ldexp(1 - 2.0 ** -24, e) for e in (-40, -3, 0, 9, 50)]
    ds += [np.ldexp(float((a << 20) + s), e - 23) for a, s, e in
           [(8, 1, 0), (9, -3, -4), (11, 5, 3), (13, -7, -10), (15, 9, 0), (12, -1, 6)]]
    return [float(np.float32(x)) for x in ds]


def test_kv_write_every_bf16_pattern_across_the_fast_range():
    """Every bf16 bit pattern as a key and a value under descales spread over
    the whole range of the division-free form and just outside it: the cache
    matches the oracle bit for bit (-0, subnormals, infinities, NaNs, quotients
    that overflow fp32 included)."""
    T, hkv, d, pool = 128, 2, 256, 3
    pat = np.arange(65536, dtype=np.uint16)
    rng = np.random.default_rng(37)
    k = torch.from_numpy(rng.permutation(pat).astype(np.int16).reshape(T, hkv, d)).view(torch.bfloat16)
    v = torch.from_numpy(rng.permutation(pat).astype(np.int16).reshape(T, hkv, d)).view(torch.bfloat16)
    slots = rng.permutation(pool * 64)[:T].astype(np.int64)
    ds = _fast_range_descales()
    for i, kd in enumerate(ds):
        vd = ds[(i + 7) % len(ds)]
        kc, vc, okc, ovc, bad = _run_both(k, v, slots, kd, vd, pool)
        assert bad == 0
        assert np.array_equal(kc, okc), (kd, np.argwhere(kc != okc)[:5])
        assert np.array_equal(vc, ovc), (vd, np.argwhere(vc != ovc)[:5])
