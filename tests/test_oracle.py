"""Pins for the CPU oracle: E4M3 codec, the Q quantizer and the attention
definition, each checked against something other than the oracle itself
(hand-worked values, closed forms, invariants, brute force, and torch's own
float8 implementation as an independent second opinion)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import bf16_bits, cu_from_lq, oracle_problem, paged_from_logical

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ALL = np.arange(256, dtype=np.uint8)
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


# ------------------------------------------------------------------ E4M3 decode

def test_e4m3_golden_codes():
    rows = []
    with open(os.path.join(GOLD, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    assert len(rows) >= 20
    got = oracle.e4m3_decode([c for c, _ in rows])
    for (c, v), g in zip(rows, got):
        if math.isnan(v):
            assert math.isnan(g), hex(c)
        else:
            assert g == v and math.copysign(1, g) == math.copysign(1, v), hex(c)


def test_e4m3_decode_matches_torch_float8():
    ref = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(ALL)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    assert np.array_equal(np.signbit(ref[m]), np.signbit(got[m]))


def test_e4m3_structure():
    v = oracle.e4m3_decode(ALL)
    assert set(np.nonzero(np.isnan(v))[0]) == {0x7F, 0xFF}
    assert np.isfinite(v[FINITE]).all() and len(FINITE) == 254
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                       # strictly monotone 0x00..0x7E
    assert np.array_equal(v[0x80:0xFF], -pos)             # sign mirror
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9
    assert np.all(np.mod(pos * 2 ** 9, 1) == 0)           # all on the 2^-9 grid


# ------------------------------------------------------------------ E4M3 encode

def test_encode_roundtrip_all_finite_codes():
    x = oracle.e4m3_decode(FINITE).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), FINITE)


def test_encode_midpoints_go_to_even_code():
    v = oracle.e4m3_decode(ALL)
    for c in range(0, 0x7E):
        for sgn in (0, 0x80):
            a, b = v[c | sgn], v[(c + 1) | sgn]
            mid = np.float32((a + b) / 2)
            assert float(mid) == (a + b) / 2
            want = (c if c % 2 == 0 else c + 1) | sgn
            assert oracle.e4m3_encode(np.array([mid]))[0] == want, (hex(c), sgn)


def test_encode_saturation_nan_zero():
    x = np.array([448, 449, 463.99, 464, 480, 1e6, np.inf, -448, -1e30, -np.inf, np.nan, -np.nan,
                  0.0, -0.0], dtype=np.float32)
    got = oracle.e4m3_encode(x)
    assert list(got) == [0x7E] * 7 + [0xFE] * 3 + [0x7F, 0xFF, 0x00, 0x80]


def test_encode_underflow():
    x = np.array([2.0 ** -10, np.nextafter(np.float32(2.0 ** -10), np.float32(1)), 3 * 2.0 ** -10,
                  2.0 ** -11, -2.0 ** -11, 2.0 ** -30], dtype=np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x00, 0x01, 0x02, 0x00, 0x80, 0x00]


def _brute_force_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by exhaustive search, ties to the even code."""
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # 0x00..0x7E, ascending
    out = np.empty(x.shape, dtype=np.uint8)
    for s in range(0, x.size, 20000):
        xs = x[s:s + 20000].astype(np.float64)
        a = np.abs(xs)
        dist = np.abs(vals[None, :] - a[:, None])
        i0 = np.argmin(dist, axis=1)
        dmin = dist[np.arange(len(a)), i0]
        i1 = np.minimum(i0 + 1, 0x7E)
        tie = (i1 != i0) & (dist[np.arange(len(a)), i1] == dmin)
        code = np.where(tie & (i0 % 2 == 1), i1, i0).astype(np.uint8)
        code = np.where(np.isinf(a), 0x7E, code)
        code = code | np.where(np.signbit(xs), 0x80, 0).astype(np.uint8)
        code = np.where(np.isnan(xs), np.where(np.signbit(xs), 0xFF, 0x7F), code)
        out[s:s + 20000] = code
    return out


def test_encode_brute_force_random():
    rng = np.random.default_rng(7)
    n = 1_000_000
    mag = np.exp2(rng.uniform(-13, 10, size=n))
    x = (mag * np.where(rng.random(n) < 0.5, -1, 1)).astype(np.float32)
    # add exact grid points and their float32 neighbours
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float32)
    mids = ((v[:-1].astype(np.float64) + v[1:]) / 2).astype(np.float32)
    extra = np.concatenate([v, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    x = np.concatenate([x, extra, -extra])
    assert np.array_equal(oracle.e4m3_encode(x), _brute_force_encode(x))


def test_encode_matches_torch_float8_in_range():
    rng = np.random.default_rng(8)
    x = (np.exp2(rng.uniform(-12, 8.7, size=200_000)) * rng.choice([-1, 1], 200_000)).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_quantize_q_is_fp32_division_then_rne():
    rng = np.random.default_rng(9)
    q = torch.from_numpy(rng.standard_normal(50_000).astype(np.float32)).to(torch.bfloat16)
    bits = bf16_bits(q)
    d = np.float32(0.0123456)
    quot = q.float().numpy() / d                      # IEEE fp32 division
    assert np.array_equal(oracle.quantize_q(bits, float(d)), _brute_force_encode(quot.astype(np.float32)))


def test_quantize_q_division_not_reciprocal_multiply():
    """Inputs built so that the exact quotient sits within an fp32 ulp of an
    E4M3 midpoint: there fl32(x / d) and fl32(x * fl32(1 / d)) round to
    different codes, and the oracle must follow the division."""
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    xs = (np.arange(0x3F00, 0x4100, 7, dtype=np.uint32) << 16).view(np.float32)
    cand_x, cand_d = [], []
    for m in mids[40:120]:
        for x in xs:
            d = np.float32(np.float64(x) / m)
            for _ in range(4):
                cand_x.append(x)
                cand_d.append(d)
                d = np.nextafter(d, np.float32(np.inf))
    cx = np.array(cand_x, np.float32)
    cd = np.array(cand_d, np.float32)
    div = cx / cd
    mul = cx * (np.float32(1) / cd)
    sel = _brute_force_encode(div) != _brute_force_encode(mul)
    assert sel.sum() >= 5, "need discriminating cases"
    bits = (cx[sel].view(np.uint32) >> 16).astype(np.uint16)
    for b, d, want in zip(bits, cd[sel], _brute_force_encode(div[sel])):
        assert oracle.quantize_q(np.array([b]), float(d))[0] == want


def test_quantize_q_nan_quotient_keeps_input_sign():
    bits = np.array([0x7FC1, 0xFFC1, 0x7F81, 0xFF81], np.uint16)       # +-qNaN, +-sNaN payloads
    assert list(oracle.quantize_q(bits, 0.5)) == [0x7F, 0xFF, 0x7F, 0xFF]
    zeros = np.array([0x0000, 0x8000], np.uint16)                     # 0 / 0 and -0 / 0
    assert list(oracle.quantize_q(zeros, 0.0)) == [0x7F, 0xFF]
    infs = np.array([0x7F80, 0xFF80], np.uint16)                      # +-inf / finite saturates
    assert list(oracle.quantize_q(infs, 3.0)) == [0x7E, 0xFE]


# ------------------------------------------------------------------ masks

def _golden_ranges():
    with open(os.path.join(GOLD, "visible_ranges.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("->")
            Lq, Lk, i, w, c = map(int, lhs.split())
            rhs = rhs.split()
            yield (Lq, Lk, i, w, c), (None if rhs == ["empty"] else (int(rhs[0]), int(rhs[1])))


def test_visible_range_golden():
    n = 0
    for args, want in _golden_ranges():
        assert oracle.visible_range(*args) == want, args
        n += 1
    assert n >= 15


def test_visible_range_brute_force():
    for Lq in (1, 2, 5, 64, 70):
        for Lk in (0, 1, 3, 63, 64, 65, 70):
            for w in (-1, 0, 1, 63, 64):
                for causal in (0, 1):
                    for i in range(Lq):
                        seen = []
                        for j in range(Lk):
                            ok = True
                            if causal and j > Lk - Lq + i:
                                ok = False
                            if w >= 0 and j < Lk - Lq + i - w:
                                ok = False
                            if ok:
                                seen.append(j)
                        want = (seen[0], seen[-1]) if seen else None
                        if seen:
                            assert seen == list(range(seen[0], seen[-1] + 1))
                        assert oracle.visible_range(Lq, Lk, i, w, causal) == want, (Lq, Lk, i, w, causal)


def test_position_one_hot_values_pin_visible_set():
    """Uniform logits (K all zero) and V[j] = e_j (one-hot on channel j): the
    output of each query row is 1/|J| on exactly the channels of its visible
    keys, and lse = ln|J|.  Runs through paging with a permuted block table."""
    rng = np.random.default_rng(11)
    D, hkv, hq = 256, 1, 2
    cases = [((5, 150), (1, 70), (64, 64), (3, 2), (2, 0)), ]
    for wl in (-1, 0, 17, 64):
        for causal in (True, False):
            for seqs in cases:
                lq = [a for a, _ in seqs]
                lk = [b for _, b in seqs]
                kl = [np.zeros((n, hkv, D), np.uint8) for n in lk]
                vl = []
                for n in lk:
                    v = np.zeros((n, hkv, D), np.uint8)
                    for j in range(n):
                        v[j, :, j] = 0x38  # 1.0
                    vl.append(v)
                kc, vc, bt = paged_from_logical(kl, vl, lk, rng)
                q = np.full((sum(lq), hq, D), 0x3F80, np.uint16)  # bf16 1.0
                prob = oracle.AttnProblem(q, False, kc, vc, bt, cu_from_lq(lq), lk, hkv, 1.0, 1.0, 1.0,
                                          1 / 16, wl, causal)
                out, lse = oracle.paged_attention(prob)
                t = 0
                for b, (Lq, Lk) in enumerate(seqs):
                    for i in range(Lq):
                        r = oracle.visible_range(Lq, Lk, i, wl, causal)
                        for h in range(hq):
                            want = np.zeros(D)
                            if r is not None:
                                want[r[0]:r[1] + 1] = 1.0 / (r[1] - r[0] + 1)
                                assert abs(lse[h, t] - math.log(r[1] - r[0] + 1)) < 1e-12
                            else:
                                assert lse[h, t] == -np.inf
                            assert np.allclose(out[t, h], want, atol=1e-14, rtol=0), (b, i, wl, causal)
                        t += 1


# ------------------------------------------------------------------ attention closed forms

def _tiny(lq, lk, hq=4, hkv=2, d=256, wl=-1, causal=True, fp8=True, seed=5):
    return synth.make_workload("t", lq, lk, hq, hkv, d, wl, causal, fp8, seed=seed)


def test_probs_sum_to_one_and_vanish_outside():
    w = _tiny([3, 70], [130, 70], wl=40)
    p = oracle_problem(w)
    for t in (0, 2, 3, 50, 72):
        for h in (0, 3):
            probs, _, _ = oracle.attention_probs(p, t, h)
            b = 0 if t < 3 else 1
            i = t if b == 0 else t - 3
            lo, hi = oracle.visible_range(int(w.lq[b]), int(w.lk[b]), i, w.window_left, w.causal)
            assert abs(probs.sum() - 1.0) < 1e-12
            assert np.all(probs[:lo] == 0) and np.all(probs[hi + 1:] == 0)
            assert np.all(probs[lo:hi + 1] > 0)


def _decoded_rows(cache, bt, b, js, hk, descale):
    return np.stack([oracle.e4m3_decode(cache[bt[b, j // 64], j % 64, hk]) * descale for j in js])


def test_identical_keys_give_mean_of_v():
    w = _tiny([4, 1], [100, 200], wl=-1, causal=True)
    p = oracle_problem(w)
    kc = p.k_cache.copy()
    kc[:, :, :, :] = kc[w.bt[0, 0], 0][None, None]  # every key row of a head = one row
    p.k_cache = np.ascontiguousarray(kc)
    out, _ = oracle.paged_attention(p)
    G = w.num_heads_q // w.num_heads_kv
    t = 0
    for b in range(w.batch):
        for i in range(int(w.lq[b])):
            lo, hi = oracle.visible_range(int(w.lq[b]), int(w.lk[b]), i, -1, True)
            for h in range(w.num_heads_q):
                v = _decoded_rows(p.v_cache, w.bt, b, range(lo, hi + 1), h // G, w.v_descale)
                assert np.allclose(out[t, h], v.mean(axis=0), rtol=1e-12, atol=1e-12)
            t += 1


def _const_problem(k_rows, v_rows, q_code=0x38, d=64, scale=1 / 8):
    """One sequence, one query, Hq = Hkv = 1, key j holds the E4M3 code k_rows[j]
    in every channel; V given per key as a full row of codes."""
    lk = len(k_rows)
    kl = [np.repeat(np.array(k_rows, np.uint8)[:, None, None], d, axis=2)]
    vl = [np.array(v_rows, np.uint8)[:, None, :]]
    kc, vc, bt = paged_from_logical(kl, vl, [lk], np.random.default_rng(3))
    q = np.full((1, 1, d), q_code, np.uint8)
    return oracle.AttnProblem(q, True, kc, vc, bt, [0, 1], [lk], 1, 1.0, 1.0, 1.0, scale, -1, True)


def test_single_key_closed_form():
    rng = np.random.default_rng(12)
    v = rng.choice(FINITE, size=(1, 64)).astype(np.uint8)
    p = _const_problem([0x40], v)      # q = 1.0, k = 2.0 in every channel
    out, lse = oracle.paged_attention(p)
    assert np.array_equal(out[0, 0], oracle.e4m3_decode(v[0]))
    assert lse[0, 0] == (1 / 8) * 64 * 2.0


def test_two_keys_logistic_closed_form():
    rng = np.random.default_rng(13)
    v = rng.choice(FINITE, size=(2, 64)).astype(np.uint8)
    p = _const_problem([0x38, 0x30], v, scale=1 / 32)  # k0 = 1.0, k1 = 0.5
    out, lse = oracle.paged_attention(p)
    s0, s1 = 64 * 1.0 / 32, 64 * 0.5 / 32
    w0 = 1 / (1 + math.exp(s1 - s0))
    want = w0 * oracle.e4m3_decode(v[0]) + (1 - w0) * oracle.e4m3_decode(v[1])
    assert np.allclose(out[0, 0], want, rtol=1e-13, atol=1e-13)
    assert abs(lse[0, 0] - np.logaddexp(s0, s1)) < 1e-13


def test_one_hot_logit_selects_v_row():
    rng = np.random.default_rng(14)
    k = [0x00] * 90
    k[37] = 0x50  # 8.0: logit 64 * 8 / 4 = 128, every other logit 0
    v = rng.choice(FINITE, size=(90, 64)).astype(np.uint8)
    p = _const_problem(k, v, scale=1 / 4)
    out, lse = oracle.paged_attention(p)
    assert np.allclose(out[0, 0], oracle.e4m3_decode(v[37]), rtol=0, atol=1e-40 + 1e-50)
    assert abs(lse[0, 0] - 128.0) < 1e-12


def test_gqa_head_mapping():
    w = _tiny([2, 1], [70, 130], hq=8, hkv=2, d=256)
    p = oracle_problem(w)
    vc = p.v_cache.copy()
    vc[:, :, 0, :] = 0x38   # KV head 0: 1.0 everywhere
    vc[:, :, 1, :] = 0x40   # KV head 1: 2.0 everywhere
    p.v_cache = np.ascontiguousarray(vc)
    p.v_descale = np.array([1.0], np.float32)
    out, _ = oracle.paged_attention(p)
    assert np.allclose(out[:, :4], 1.0, rtol=0, atol=1e-13) and np.allclose(out[:, 4:], 2.0, rtol=0, atol=1e-13)


def test_descale_scaling_is_exact():
    w = _tiny([3, 2], [90, 65], wl=20)
    p = oracle_problem(w)
    o1, l1 = oracle.paged_attention(p)
    p2 = oracle_problem(w, v_descale=np.float32(w.v_descale * 2))
    o2, l2 = oracle.paged_attention(p2)
    assert np.array_equal(o2, 2 * o1) and np.array_equal(l1, l2)
    p3 = oracle_problem(w, k_descale=np.float32(w.k_descale * 2))
    p4 = oracle_problem(w, softmax_scale=np.float32(w.softmax_scale * 2))
    o3, l3 = oracle.paged_attention(p3)
    o4, l4 = oracle.paged_attention(p4)
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)
    # E4M3 Q: doubling q_descale is the same as doubling the softmax scale
    p6 = oracle_problem(w, q_descale=np.float32(w.q_descale * 2))
    o6, l6 = oracle.paged_attention(p6)
    assert np.array_equal(o6, o4) and np.array_equal(l6, l4)
    assert not np.array_equal(o6, o1)
    # per-(batch, kv head) descales: doubling only sequence 1's V doubles only its rows
    kd = np.full((2, 2), w.k_descale, np.float32)
    vd = np.full((2, 2), w.v_descale, np.float32)
    vd[1, :] *= 2
    p5 = oracle_problem(w, k_descale=kd.ravel(), v_descale=vd.ravel(), descale_batch_stride=2,
                        descale_head_stride=1)
    o5, _ = oracle.paged_attention(p5)
    assert np.array_equal(o5[:3], o1[:3]) and np.array_equal(o5[3:], 2 * o1[3:])


def test_page_permutation_invariance():
    w = _tiny([2, 5], [200, 150], wl=70)
    p = oracle_problem(w)
    o1, l1 = oracle.paged_attention(p)
    rng = np.random.default_rng(15)
    perm = rng.permutation(p.k_cache.shape[0])   # new position of each old page
    kc = np.empty_like(p.k_cache)
    vc = np.empty_like(p.v_cache)
    kc[perm] = p.k_cache
    vc[perm] = p.v_cache
    p2 = oracle_problem(w, k_cache=kc, v_cache=vc, block_table=perm[w.bt].astype(np.int32))
    o2, l2 = oracle.paged_attention(p2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_poison_outside_visible_does_not_leak():
    w = _tiny([3, 1], [300, 260], wl=50)
    p = oracle_problem(w)
    assert (p.k_cache[w.poison_page] == 0x7F).all()
    o1, l1 = oracle.paged_attention(p)
    assert np.isfinite(o1).all() and np.isfinite(l1).all()
    # replacing the poison with finite bytes changes nothing
    kc, vc = p.k_cache.copy(), p.v_cache.copy()
    kc[kc == 0x7F] = 0x11
    vc[vc == 0x7F] = 0x22
    o2, l2 = oracle.paged_attention(oracle_problem(w, k_cache=kc, v_cache=vc))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_empty_rows():
    w = _tiny([5, 2], [3, 0], hq=2, hkv=1, d=64, causal=True)
    out, lse = oracle.paged_attention(oracle_problem(w))
    # seq 0: queries 0, 1 sit at p = -2, -1 -> nothing visible; seq 1 has no keys
    for t in (0, 1, 5, 6):
        assert np.all(out[t] == 0) and np.all(lse[:, t] == -np.inf)
    for t in (2, 3, 4):
        assert np.isfinite(lse[:, t]).all()


def test_bf16_q_path_reads_bf16_exactly():
    d = 64
    kl = [np.full((1, 1, d), 0x38, np.uint8)]          # k = 1.0
    vl = [np.full((1, 1, d), 0x40, np.uint8)]
    kc, vc, bt = paged_from_logical(kl, vl, [1], np.random.default_rng(4))
    q = np.full((1, 1, d), 0x3FC0, np.uint16)           # bf16 1.5
    p = oracle.AttnProblem(q, False, kc, vc, bt, [0, 1], [1], 1, 123.0, 1.0, 1.0, 0.5, -1, True)
    out, lse = oracle.paged_attention(p)
    assert lse[0, 0] == 0.5 * 1.5 * d                   # q_descale is not applied to bf16 Q
    assert np.all(out == 2.0)


def test_bad_page_id_is_refused():
    w = _tiny([1], [70], hq=2, hkv=1, d=64)
    bt = w.bt.copy()
    bt[0, 1] = 10_000
    with pytest.raises(ValueError):
        oracle.paged_attention(oracle_problem(w, block_table=bt))


def test_tiny_prefill_config_is_finite():
    w = synth.make_config("tiny_prefill_hd256")
    out, lse = oracle.paged_attention(oracle_problem(w))
    assert out.shape == (256, 4, 256) and np.isfinite(out).all() and np.isfinite(lse).all()


# ------------------------------------------------------------------ KV-cache write

def _bf16_from_f32(a):
    """Exact bf16 bit patterns of float32 values that bf16 represents exactly."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    assert np.all(u & 0xFFFF == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def _write_case(seed, T=40, hkv=2, d=16, pages=6, pad_every=5):
    rng = np.random.default_rng(seed)
    slots = rng.permutation(pages * oracle.PAGE)[:T].astype(np.int64)
    slots[::pad_every] = -1
    return rng, slots


def test_kv_write_roundtrip_of_exact_codes_lands_in_slot_order():
    # x = decode(c) * 2^-3 is exact in bf16 and x / 2^-3 = decode(c), so every
    # finite code must come back unchanged, at its token's slot
    rng, slots = _write_case(1)
    T, hkv, d, pages = 40, 2, 16, 6
    codes = rng.choice(FINITE, size=(T, hkv, d))
    codes_v = rng.choice(FINITE, size=(T, hkv, d))
    ds = 0.125
    k = _bf16_from_f32(oracle.e4m3_decode(codes) * ds)
    v = _bf16_from_f32(oracle.e4m3_decode(codes_v) * ds)
    kc = np.full((pages, 64, hkv, d), 0x7F, np.uint8)
    vc = np.full((pages, 64, hkv, d), 0x7F, np.uint8)
    assert oracle.kv_cache_write(k, v, slots, ds, ds, kc, vc) == 0
    flat_k, flat_v = kc.reshape(-1, hkv, d), vc.reshape(-1, hkv, d)
    written = np.zeros(pages * 64, bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        written[slots[t]] = True
        assert np.array_equal(flat_k[slots[t]], codes[t]), t
        assert np.array_equal(flat_v[slots[t]], codes_v[t]), t
    assert np.all(flat_k[~written] == 0x7F) and np.all(flat_v[~written] == 0x7F)


def test_kv_write_then_attention_matches_directly_paged_cache():
    # a sequence written token by token into scattered slots, read back through a
    # block table of those pages by the attention oracle, equals the same codes
    # laid out by the independent test helper
    rng = np.random.default_rng(2)
    Lk, hkv, d, G = 150, 2, 32, 2
    n_pages = (Lk + 63) // 64
    pool = 9
    phys = rng.permutation(pool)[:n_pages]
    slots = np.array([phys[t // 64] * 64 + t % 64 for t in range(Lk)], np.int64)
    ds_k, ds_v = 0.25, 0.5
    ck = rng.choice(FINITE, size=(Lk, hkv, d))
    cv = rng.choice(FINITE, size=(Lk, hkv, d))
    k = _bf16_from_f32(oracle.e4m3_decode(ck) * ds_k)
    v = _bf16_from_f32(oracle.e4m3_decode(cv) * ds_v)
    kc = np.full((pool, 64, hkv, d), 0x7F, np.uint8)
    vc = np.full((pool, 64, hkv, d), 0x7F, np.uint8)
    order = rng.permutation(Lk)
    assert oracle.kv_cache_write(k[order], v[order], slots[order], ds_k, ds_v, kc, vc) == 0
    bt = np.full((1, n_pages), pool - 1, np.int32)
    bt[0, :] = phys
    q = rng.normal(size=(3, hkv * G, d)).astype(np.float32)
    qb = _bf16_from_f32(q.astype(np.float32).view(np.uint32).__and__(0xFFFF0000).view(np.float32))
    common = dict(q=qb, q_is_e4m3=False, cu_seqlens_q=np.array([0, 3], np.int32), seqused_k=np.array([Lk], np.int32),
                  num_heads_kv=hkv, q_descale=1.0, k_descale=ds_k, v_descale=ds_v, softmax_scale=0.2,
                  window_left=-1, causal=True)
    got, lse_got = oracle.paged_attention(oracle.AttnProblem(k_cache=kc, v_cache=vc, block_table=bt, **common))
    kc2, vc2, bt2 = paged_from_logical([ck], [cv], [Lk], np.random.default_rng(3))
    want, lse_want = oracle.paged_attention(oracle.AttnProblem(k_cache=kc2, v_cache=vc2, block_table=bt2, **common))
    assert np.array_equal(got, want) and np.array_equal(lse_got, lse_want)


def test_kv_write_padding_slots_write_nothing():
    rng = np.random.default_rng(4)
    T, hkv, d, pages = 12, 1, 8, 2
    k = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    kc = np.full((pages, 64, hkv, d), 0x5A, np.uint8)
    vc = np.full((pages, 64, hkv, d), 0x5A, np.uint8)
    assert oracle.kv_cache_write(k, k, np.full(T, -1, np.int64), 1.0, 1.0, kc, vc) == 0
    assert np.all(kc == 0x5A) and np.all(vc == 0x5A)


def test_kv_write_is_independent_of_token_order():
    rng, slots = _write_case(5)
    T, hkv, d, pages = 40, 2, 16, 6
    k = _bf16_from_f32(rng.normal(size=(T, hkv, d)).astype(np.float32).view(np.uint32).__and__(0xFFFF0000)
                       .view(np.float32))
    v = _bf16_from_f32(rng.normal(size=(T, hkv, d)).astype(np.float32).view(np.uint32).__and__(0xFFFF0000)
                       .view(np.float32))
    a = [np.zeros((pages, 64, hkv, d), np.uint8) for _ in range(4)]
    oracle.kv_cache_write(k, v, slots, 0.03, 0.07, a[0], a[1])
    p = rng.permutation(T)
    oracle.kv_cache_write(k[p], v[p], slots[p], 0.03, 0.07, a[2], a[3])
    assert np.array_equal(a[0], a[2]) and np.array_equal(a[1], a[3])


def test_kv_write_codes_are_nearest_e4m3_of_fp32_quotient():
    # brute force: each written code decodes to a finite E4M3 value nearest to
    # fl32(x / descale) (ties to the even code, |quotient| >= 464 saturates to 448)
    rng = np.random.default_rng(6)
    T, hkv, d = 64, 1, 16
    x = (rng.normal(size=(T, hkv, d)) * rng.choice([1e-3, 1, 40, 3000], size=(T, 1, 1))).astype(np.float32)
    kb = _bf16_from_f32(x.view(np.uint32).__and__(0xFFFF0000).view(np.float32))
    ds = np.float32(0.37)
    kc = np.zeros((1, 64, hkv, d), np.uint8)
    vc = np.zeros_like(kc)
    oracle.kv_cache_write(kb, kb, np.arange(T, dtype=np.int64), float(ds), float(ds), kc, vc)
    vals = oracle.e4m3_decode(FINITE)
    xs = (kb.astype(np.uint32) << 16).view(np.float32)
    quot = (xs.astype(np.float64) / np.float64(ds)).astype(np.float32).astype(np.float64).reshape(-1)
    got = kc.reshape(-1)
    for qv, c in zip(quot, got):
        dist = np.abs(vals - np.clip(qv, -448.0, 448.0))
        best = dist.min()
        assert abs(oracle.e4m3_decode([c])[0] - np.clip(qv, -448.0, 448.0)) == best
        if (dist == best).sum() > 1 and qv != 0:
            assert int(c) & 1 == 0, (qv, hex(c))


def test_kv_write_counts_and_skips_slots_past_the_cache():
    rng = np.random.default_rng(7)
    T, hkv, d, pages = 6, 1, 8, 1
    k = rng.integers(0, 0x3F00, size=(T, hkv, d), dtype=np.uint16)
    slots = np.array([0, 64, 5, 1000, -1, 63], np.int64)
    kc = np.full((pages, 64, hkv, d), 0x11, np.uint8)
    vc = np.full_like(kc, 0x11)
    assert oracle.kv_cache_write(k, k, slots, 1.0, 1.0, kc, vc) == 2
    untouched = [s for s in range(64) if s not in (0, 5, 63)]
    assert np.all(kc[0, untouched] == 0x11)


def test_kv_write_reads_strided_token_rows():
    rng = np.random.default_rng(8)
    T, hkv, d, pages = 20, 2, 8, 1
    wide = rng.integers(0, 0x3F00, size=(T, 3 * hkv * d), dtype=np.uint16)
    k = wide[:, hkv * d:2 * hkv * d]
    v = wide[:, 2 * hkv * d:]
    slots = rng.permutation(64)[:T].astype(np.int64)
    a = [np.zeros((pages, 64, hkv, d), np.uint8) for _ in range(4)]
    oracle.kv_cache_write(k, v, slots, 0.5, 0.25, a[0], a[1])
    oracle.kv_cache_write(np.ascontiguousarray(k), np.ascontiguousarray(v), slots, 0.5, 0.25, a[2], a[3])
    assert np.array_equal(a[0], a[2]) and np.array_equal(a[1], a[3])


# ------------------------------------------------------------------ LSE combine

def _to_bf16_bits(a):
    """Round fp64 values to bf16 (round to nearest even) and return the bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def _noncausal_problem(seed, lk, hkv=2, G=2, d=32, lq=3):
    rng = np.random.default_rng(seed)
    kl = [rng.choice(FINITE[FINITE < 0x70], size=(n, hkv, d)) for n in lk]
    vl = [rng.choice(FINITE[FINITE < 0x70], size=(n, hkv, d)) for n in lk]
    q = _to_bf16_bits(rng.normal(size=(lq * len(lk), hkv * G, d)))
    return rng, kl, vl, q


def _attend(q, kl, vl, lk, lq, hkv, seed):
    kc, vc, bt = paged_from_logical(kl, vl, lk, np.random.default_rng(seed))
    prob = oracle.AttnProblem(q=q, q_is_e4m3=False, k_cache=kc, v_cache=vc, block_table=bt,
                              cu_seqlens_q=cu_from_lq([lq] * len(lk)), seqused_k=np.array(lk, np.int32),
                              num_heads_kv=hkv, q_descale=1.0, k_descale=0.5, v_descale=0.25, softmax_scale=0.3,
                              window_left=-1, causal=False)
    return oracle.paged_attention(prob)


def test_lse_combine_of_key_shards_is_the_whole_softmax():
    # attention over two disjoint key shards, each returned as bf16 O and f32 LSE,
    # combines to the attention over all keys (within the bf16 rounding of the parts)
    lk, lq, hkv = [150, 70], 3, 2
    rng, kl, vl, q = _noncausal_problem(21, lk, hkv=hkv, lq=lq)
    full, lse_full = _attend(q, kl, vl, lk, lq, hkv, 1)
    cut = [64, 64]
    a, la = _attend(q, [k[:c] for k, c in zip(kl, cut)], [v[:c] for v, c in zip(vl, cut)], cut, lq, hkv, 2)
    rest = [n - c for n, c in zip(lk, cut)]
    b, lb = _attend(q, [k[c:] for k, c in zip(kl, cut)], [v[c:] for v, c in zip(vl, cut)], rest, lq, hkv, 3)
    parts = np.stack([_to_bf16_bits(a), _to_bf16_bits(b)])
    lses = np.stack([la, lb]).astype(np.float32)
    out, lse = oracle.lse_combine(parts, lses)
    scale = np.abs(full).max()
    assert np.abs(out - full).max() <= 2.0 ** -8 * scale
    assert np.abs(lse - lse_full).max() <= 1e-5


def test_lse_combine_single_part_and_two_equal_parts():
    rng = np.random.default_rng(22)
    o = _to_bf16_bits(rng.normal(size=(1, 5, 4, 16)))
    l = rng.normal(size=(1, 4, 5)).astype(np.float32)
    out, lse = oracle.lse_combine(o, l)
    dec = (o[0].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(out, dec.astype(np.float64)) and np.array_equal(lse, l[0].astype(np.float64))
    # two parts with the same LSE c: L = c + ln 2, O = (O1 + O2) / 2
    o2 = _to_bf16_bits(rng.normal(size=(2, 5, 4, 16)))
    l2 = np.repeat(l, 2, axis=0)
    out, lse = oracle.lse_combine(o2, l2)
    d2 = (o2.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(out, (d2[0] + d2[1]) / 2, rtol=0, atol=1e-12)
    assert np.allclose(lse, l[0].astype(np.float64) + math.log(2.0), rtol=0, atol=1e-12)


def test_lse_combine_empty_parts():
    rng = np.random.default_rng(23)
    o = _to_bf16_bits(rng.normal(size=(3, 4, 2, 8)))
    l = rng.normal(size=(3, 2, 4)).astype(np.float32)
    l[1] = -np.inf              # an empty shard adds nothing
    out, lse = oracle.lse_combine(o, l)
    out2, lse2 = oracle.lse_combine(o[[0, 2]], l[[0, 2]])
    assert np.allclose(out, out2, rtol=0, atol=1e-14) and np.allclose(lse, lse2, rtol=0, atol=1e-14)
    l[:] = -np.inf              # no key anywhere: O = 0, lse = -inf
    out, lse = oracle.lse_combine(o, l)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_lse_combine_is_independent_of_part_order():
    rng = np.random.default_rng(24)
    o = _to_bf16_bits(rng.normal(size=(4, 6, 2, 8)))
    l = (rng.normal(size=(4, 2, 6)) * 5).astype(np.float32)
    a = oracle.lse_combine(o, l)
    p = [2, 0, 3, 1]
    b = oracle.lse_combine(o[p], l[p])
    assert np.allclose(a[0], b[0], rtol=0, atol=1e-12) and np.allclose(a[1], b[1], rtol=0, atol=1e-12)


# ------------------------------------------------------------------ attention sinks

def _sink_problem(seed, sinks, lq=(3, 1, 4), lk=(70, 1, 130), window_left=-1, causal=True):
    rng = np.random.default_rng(seed)
    hkv, G, d = 2, 2, 16
    kl = [rng.choice(FINITE[FINITE < 0x70], size=(n, hkv, d)) for n in lk]
    vl = [rng.choice(FINITE[FINITE < 0x70], size=(n, hkv, d)) for n in lk]
    kc, vc, bt = paged_from_logical(kl, vl, list(lk), np.random.default_rng(seed + 1))
    q = _to_bf16_bits(rng.normal(size=(sum(lq), hkv * G, d)))
    return oracle.AttnProblem(q=q, q_is_e4m3=False, k_cache=kc, v_cache=vc, block_table=bt,
                              cu_seqlens_q=cu_from_lq(list(lq)), seqused_k=np.array(lk, np.int32), num_heads_kv=hkv,
                              q_descale=1.0, k_descale=0.5, v_descale=0.25, softmax_scale=0.3,
                              window_left=window_left, causal=causal, sinks=sinks)


def test_sinks_at_minus_inf_change_nothing():
    a = oracle.paged_attention(_sink_problem(41, None))
    b = oracle.paged_attention(_sink_problem(41, np.full(4, -np.inf, np.float32)))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_sink_is_an_extra_logit_with_no_value():
    # o_sink = o * exp(lse - lse_sink), lse_sink = ln(exp(lse) + exp(sink)), row by row
    sinks = np.array([0.5, -2.0, 3.0, 8.0], np.float32)
    o, lse = oracle.paged_attention(_sink_problem(42, None))
    os_, lses = oracle.paged_attention(_sink_problem(42, sinks))
    want_lse = np.logaddexp(lse, sinks[:, None].astype(np.float64))
    assert np.allclose(lses, want_lse, rtol=0, atol=1e-12)
    assert np.allclose(os_, o * np.exp(lse - want_lse).T[:, :, None], rtol=0, atol=1e-12)


def test_sink_closed_form_single_key():
    # one visible key with logit s0 (= the sinkless lse) and value v0 (= the sinkless output):
    # o = v0 * sigmoid(s0 - c), lse = ln(e^s0 + e^c)
    sinks = np.array([1.0, -1.0, 0.0, 2.5], np.float32)
    o, lse = oracle.paged_attention(_sink_problem(43, None, lq=(1,), lk=(1,), causal=False))
    os_, lses = oracle.paged_attention(_sink_problem(43, sinks, lq=(1,), lk=(1,), causal=False))
    c = sinks.astype(np.float64)
    s0 = lse[:, 0]
    sig = 1.0 / (1.0 + np.exp(c - s0))
    assert np.allclose(lses[:, 0], np.log(np.exp(s0) + np.exp(c)), rtol=0, atol=1e-12)
    assert np.allclose(os_[0], o[0] * sig[:, None], rtol=0, atol=1e-12)


def test_sink_on_a_row_with_no_visible_key():
    # window_left = 0 and a query before every key: nothing visible, o = 0 and lse = sink
    sinks = np.array([0.25, -3.0, 1.5, 0.0], np.float32)
    prob = _sink_problem(44, sinks, lq=(2,), lk=(1,), causal=True)
    o, lse = oracle.paged_attention(prob)
    assert np.all(o[0] == 0) and np.array_equal(lse[:, 0], sinks.astype(np.float64))
