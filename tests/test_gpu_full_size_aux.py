"""The KV-cache write and the LSE combine at the full sizes the bench times,
against the oracle: every byte of both paged caches (written slots and the
poison left around them) for the mixed batch's 8128 new tokens at head dim 256
and 512, and every merged row of the two-shard combine of that batch's 8128 x
32 query rows at head dim 512."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("name", synth.KV_WRITE_CONFIG_NAMES)
def test_kv_write_full_size_bit_exact(name):
    import fp8_paged_attention_gb300 as fp8pa
    w = synth.make_kv_write_config(name)
    shape = (w.num_pages, synth.PAGE, w.num_heads_kv, w.head_dim)
    kc = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda")
    vc = torch.full_like(kc, 0x7F)
    kd = torch.tensor([w.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([w.v_descale], dtype=torch.float32, device="cuda")
    slots = w.slot_mappings[0]
    fp8pa.kv_cache_write(w.key.cuda(), w.value.cuda(), kc, vc, slots.cuda(), kd, vd)
    okc = np.full(shape, 0x7F, np.uint8)
    ovc = np.full(shape, 0x7F, np.uint8)
    bad = oracle.kv_cache_write(_bits(w.key), _bits(w.value), slots.numpy(), w.k_descale, w.v_descale, okc, ovc)
    assert bad == 0
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)


def test_lse_combine_full_size_matches_oracle():
    import fp8_paged_attention_gb300 as fp8pa
    w = synth.make_combine_config("lse_combine_mixed_hd512")
    got, got_lse = fp8pa.lse_combine(w.o_parts.cuda(), w.lse_parts.cuda())
    want, want_lse = oracle.lse_combine(_bits(w.o_parts), w.lse_parts.numpy())
    g = got.float().cpu().numpy()
    # bf16 output: half an ulp of the merged value, relative to max(1, |value|)
    err = np.abs(g - want) / np.maximum(1.0, np.abs(want))
    assert err.max() <= 4e-3, err.max()
    gl = got_lse.cpu().numpy()
    assert np.abs(gl - want_lse).max() <= 1e-5 * max(1.0, np.abs(want_lse).max())
