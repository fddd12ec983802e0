"""Host-side tests of the C ABI: the library loads, exports every declared
entry point, and rejects bad arguments before touching the GPU; workspace and
split sizing are pure functions of host-known sizes."""
import ctypes
import os
import re

import pytest
import torch

import fp8_paged_attention_gb300 as fp8pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions(header="fp8pa.h"):
    txt = open(os.path.join(ROOT, "include", header)).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|void|const char\*)\s+(\w+)\s*\(", txt, flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = fp8pa.load_library()
    names = _declared_functions()
    assert {"fp8_paged_attn_fwd", "quantize_q_fp8", "fp8pa_workspace_size"} <= set(names)
    hooks = _declared_functions("fp8pa_testing.h")
    assert {"fp8pa_set_wait_limit", "fp8pa_set_bf16_dequant_v"} <= set(hooks)
    for n in names + hooks:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_product_header_has_no_process_wide_switch():
    # tuning and test hooks live in fp8pa_testing.h, not in the product interface
    assert not [n for n in _declared_functions() if n.startswith("fp8pa_set_")]


def _fwd(**kw):
    lib = fp8pa.load_library()
    a = dict(q=16, q_dtype=1, k=16, v=16, num_pages=4, bt=16, max_pages=4, cu=16, su=16, batch=2, total_q=2,
             max_seqlen_q=1, hq=32, hkv=16, d=256, qd=16, kd=16, vd=16, sb=0, sh=0, scale=0.0625, wl=-1,
             causal=1, splits=0, ws=256, ws_bytes=1 << 30, out=16, lse=0, stream=0)
    a.update(kw)
    return lib.fp8_paged_attn_fwd(*a.values())


@pytest.mark.parametrize("kw,code,needle", [
    (dict(d=128), 2, "head_dim 128"),
    (dict(d=256, q_dtype=0), 2, "bfloat16"),
    (dict(q_dtype=7), 1, "q_dtype"),
    (dict(hq=30, hkv=16), 2, "multiple"),
    (dict(hq=96, hkv=3), 2, "per KV head"),
    (dict(batch=-1), 1, ">= 0"),
    (dict(wl=-2), 1, "window_left"),
    (dict(splits=-1), 1, "num_splits"),
    (dict(max_pages=0), 1, "max_pages"),
    (dict(causal=2), 1, "causal"),
    (dict(q=0), 1, "null"),
    (dict(k=8), 1, "aligned"),
    (dict(ws_bytes=16), 1, "workspace too small"),
    (dict(ws=128), 1, "256-byte"),
    (dict(scale=float("inf")), 1, "finite"),
    (dict(sb=-1), 1, "strides"),
    (dict(num_pages=0), 1, "num_pages"),
])
def test_fwd_rejects_bad_arguments_before_launch(kw, code, needle):
    rc = _fwd(**kw)
    assert rc == code
    assert needle in fp8pa.load_library().fp8pa_last_error().decode()


def test_empty_batch_is_a_noop():
    assert _fwd(batch=0, total_q=0, max_seqlen_q=0) == 0


def test_quantize_rejects_bad_arguments():
    lib = fp8pa.load_library()
    assert lib.quantize_q_fp8(16, 16, 16, -1, 0) == 1
    assert lib.quantize_q_fp8(0, 16, 16, 8, 0) == 1
    assert lib.quantize_q_fp8(0, 0, 0, 0, 0) == 0


def test_workspace_and_splits_are_host_functions():
    E4M3, BF16 = fp8pa.FP8PA_E4M3, fp8pa.FP8PA_BF16
    # SWA decode: 64 x 1 query, Hq 32 / Hkv 16, D 256, window 1023, 144 pages
    ws = fp8pa.workspace_size(64, 64, 1, 32, 16, 256, E4M3, 144, 1023, 0)
    s = fp8pa.num_splits(64, 64, 1, 32, 16, 256, E4M3, 144, 1023, 0)
    assert ws > 0 and 1 <= s <= 64
    assert ws == fp8pa.workspace_size(64, 64, 1, 32, 16, 256, E4M3, 144, 1023, 0)
    # explicit split count is honoured and grows the workspace by the partial buffers
    w1 = fp8pa.workspace_size(64, 64, 1, 32, 4, 512, BF16, 144, -1, 1)
    w4 = fp8pa.workspace_size(64, 64, 1, 32, 4, 512, BF16, 144, -1, 4)
    assert fp8pa.num_splits(64, 64, 1, 32, 4, 512, BF16, 144, -1, 4) == 4
    assert w4 - w1 >= 4 * 64 * 32 * 512 * 4
    # fewer (sequence, KV head) units than SMs: long contexts get split; plenty of units: no split
    assert fp8pa.num_splits(8, 8, 1, 32, 4, 512, BF16, 144, -1, 0) > 1
    assert fp8pa.num_splits(8, 8, 1, 32, 4, 512, E4M3, 144, -1, 0) > 1
    assert fp8pa.num_splits(64, 64, 1, 32, 4, 512, E4M3, 144, -1, 0) == 1
    # 32-row tiles (4 verify tokens x 8 heads) with 1-4 waves of long units: the split count whose
    # item waves fill the last one best, with a 2 % cost per extra split (64 x 4 units on 152 SMs:
    # 4 splits, 6.7 waves).  The SM count is the visible device's (152 on GB300, and without a device).
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    units = 64 * 4
    if sms <= units < 4 * sms:
        costs = {s: -(-units * s // sms) / s * (1 + 0.02 * (s - 1)) for s in range(1, 9)}
        expect = min(costs, key=lambda s: (costs[s], s))
        assert fp8pa.num_splits(64, 256, 4, 32, 4, 512, BF16, 448, -1, 0) == expect
        if sms == 152:
            assert expect == 4
    assert fp8pa.num_splits(64, 256, 4, 32, 4, 512, BF16, 448, -1, 0) > 1
    # 16-row decode tiles with as many units stay whole, and so do 32-row tiles past four waves
    assert fp8pa.num_splits(64, 64, 1, 32, 4, 512, BF16, 144, -1, 0) == 1
    assert fp8pa.num_splits(160, 640, 4, 32, 4, 512, BF16, 448, -1, 0) == 1
    # the mixed chunked-prefill batch has plenty of units: no split
    assert fp8pa.num_splits(4033, 8128, 4096, 32, 16, 256, E4M3, 128, 1023, 0) == 1
    # launches: plan + attention (+ combine when split)
    assert fp8pa.kernel_launches(4033, 8128, 4096, 32, 16, 256, E4M3, 128, 1023, 0) == 3  # two row classes
    assert fp8pa.kernel_launches(64, 64, 1, 32, 4, 512, BF16, 144, -1, 1) == 2
    # rejected shapes size to 0
    assert fp8pa.workspace_size(1, 1, 1, 32, 16, 128, E4M3, 4, -1, 0) == 0
    assert fp8pa.workspace_size(1, 1, 1, 32, 16, 256, BF16, 4, -1, 0) == 0
    assert fp8pa.num_splits(1, 1, 1, 30, 16, 256, E4M3, 4, -1, 0) == 0


def _kvw(**kw):
    import fp8_paged_attention_gb300 as fp8pa
    lib = fp8pa.load_library()
    a = dict(key=16, value=16, ks=256, vs=256, kc=8, vc=8, pages=4, slots=8, T=3, hkv=1, d=256, kd=4, vd=4)
    a.update(kw)
    return lib.fp8pa_kv_cache_write(a["key"], a["value"], a["ks"], a["vs"], a["kc"], a["vc"], a["pages"], a["slots"],
                                    a["T"], a["hkv"], a["d"], a["kd"], a["vd"], None)


@pytest.mark.parametrize("kw", [dict(key=0), dict(slots=0), dict(kd=0), dict(T=-1), dict(hkv=0), dict(d=6),
                                dict(ks=255), dict(vs=8), dict(key=24), dict(kc=4)])
def test_kv_cache_write_rejects_bad_arguments_before_launch(kw):
    # every check runs on the host before any device access (the pointers here are not device memory)
    assert _kvw(**kw) == 1  # FP8PA_EINVAL


def test_kv_cache_write_zero_tokens_is_a_noop():
    assert _kvw(T=0) == 0


@pytest.mark.parametrize("args", [(0, 16, 2, 4, 8, 64, 16, 16), (16, 0, 2, 4, 8, 64, 16, 16), (16, 16, 0, 4, 8, 64, 16, 16),
                                  (16, 16, 2, -1, 8, 64, 16, 16), (16, 16, 2, 4, 8, 60, 16, 16),
                                  (24, 16, 2, 4, 8, 64, 16, 16), (16, 16, 2, 4, 8, 64, 8, 16)])
def test_lse_combine_rejects_bad_arguments_before_launch(args):
    lib = fp8pa.load_library()
    o, l, p, t, h, d, out, lo = args
    assert lib.fp8pa_lse_combine(o, l, p, t, h, d, out, lo, None) == 1  # FP8PA_EINVAL


def test_lse_combine_zero_tokens_is_a_noop():
    assert fp8pa.load_library().fp8pa_lse_combine(16, 16, 2, 0, 8, 64, 16, 16, None) == 0
