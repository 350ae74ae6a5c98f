"""kv_state_get / kv_state_set on the GPU: stream bytes bit-exact with the oracle,
layout-independent, byte-identical round trips, and rejected streams write nothing."""

import numpy as np
import pytest
import torch

import seeded_inputs as si
from golden_io import read_hex
from oracle import state as ostate
from parity_util import assert_cache_equal
from test_gpu_append import run_appends

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
@pytest.mark.parametrize("shape", [(3, 8, 128), (1, 2, 64), (2, 1, 32), (2, 3, 96)])
def test_pack_matches_oracle_and_restores_across_layouts(kvc, cache_type, shape):
    n_layer, H, D = shape
    w = si.small_workload("st", H, H, D, cache_type, "bf16", n_prompt=61, chunk=20, n_decode=2, seed=D + H,
                          n_layer=n_layer)
    n = w.n_tokens
    for src_layout, dst_layout in (("head_major", "layer_major"), ("layer_major", "head_major")):
        g, o = run_appends(kvc, w, src_layout)
        blob = kvc.kv_state_get(g, n)
        torch.cuda.synchronize()
        ref = ostate.pack(o, n)
        assert blob.numel() == ref.size
        assert np.array_equal(blob.cpu().numpy(), ref)
        g2 = kvc.KVCache(w.n_layer, w.n_ctx, H, D, cache_type, dst_layout)
        assert kvc.kv_state_set(g2, blob) == n
        torch.cuda.synchronize()
        assert_cache_equal(g2, o, n)
        assert np.array_equal(kvc.kv_state_get(g2, n).cpu().numpy(), ref)
        # a prefix of the positions
        assert np.array_equal(kvc.kv_state_get(g, 17).cpu().numpy(), ostate.pack(o, 17))


def test_empty_state(kvc):
    g = kvc.KVCache(2, 16, 2, 64, "q8_0")
    blob = kvc.kv_state_get(g, 0)
    assert blob.numel() == 32
    assert kvc.kv_state_set(g, blob) == 0


@pytest.mark.parametrize("fixture,cache_type,n", [("state_q8_0_tiny.txt", "q8_0", 2), ("state_f16_tiny.txt", "f16", 1)])
def test_hand_written_fixture_round_trips(kvc, fixture, cache_type, n):
    ref = read_hex(fixture)
    for layout in ("head_major", "layer_major"):
        g = kvc.KVCache(1, 4, 1, 32, cache_type, layout)
        assert kvc.kv_state_set(g, torch.from_numpy(ref).cuda()) == n
        assert np.array_equal(kvc.kv_state_get(g, n).cpu().numpy(), ref)
    if cache_type == "q8_0":
        assert g.codes(0)[0, 0, 0].cpu().tolist() == [-127] + list(range(-15, 16))
        assert g.codes(1)[0, 1, 0, :6].cpu().tolist() == [127, 1, -1, 2, -3, 0]


@pytest.mark.parametrize("mutate", ["magic", "version", "shape", "type", "tokens", "reserved", "size"])
def test_rejected_state_writes_nothing(kvc, mutate):
    w = si.small_workload("bad", 2, 2, 64, "q8_0", "bf16", n_prompt=20, chunk=20, n_decode=0, seed=3)
    g, _ = run_appends(kvc, w, "head_major")
    blob = kvc.kv_state_get(g, 20).cpu().numpy().copy()
    words = blob[:32].view("<u4")
    if mutate == "magic":
        words[0] ^= 1
    elif mutate == "version":
        words[1] = 2
    elif mutate == "shape":
        words[4] = 128
    elif mutate == "type":
        words[5] = 0
    elif mutate == "tokens":
        words[6] = w.n_ctx + 1
    elif mutate == "reserved":
        words[7] = 5
    elif mutate == "size":
        blob = blob[:-16]
    dst = kvc.KVCache(w.n_layer, w.n_ctx, 2, 64, "q8_0", "layer_major")
    for kv in (0, 1):
        dst.codes(kv).fill_(3)
        dst.scales(kv).fill_(0.25)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kv_state_set(dst, torch.from_numpy(blob).cuda())
    assert e.value.status == kvc.KVC_EFORMAT
    torch.cuda.synchronize()
    for kv in (0, 1):
        assert (dst.codes(kv).cpu() == 3).all() and (dst.scales(kv).cpu() == 0.25).all()
