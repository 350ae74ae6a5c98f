"""decode_attn on the GPU: within tolerance of the oracle; bitwise equal across layouts."""

import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity_util import assert_close, np32
from test_gpu_append import run_appends

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


CASES = [
    # H_q, H_kv, D, cache, in dtype, tokens
    (40, 8, 128, "q8_0", "bf16", 700),
    (40, 8, 128, "f16", "bf16", 700),
    (4, 2, 64, "q8_0", "f32", 300),
    (4, 2, 64, "f16", "f16", 300),
    (8, 8, 128, "q8_0", "bf16", 150),   # G = 1
    (16, 1, 64, "q8_0", "bf16", 200),   # G = 16
    (24, 2, 128, "f16", "bf16", 90),    # G = 12: heads in both row halves of the MMA
    (32, 2, 128, "q8_0", "f32", 333),   # G = 16 at head_dim 128: every padded head column in use
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%d-%d-%d-%s-%s" % c[:5])
def test_decode_matches_oracle(kvc, case):
    hq, hkv, d, cache, dt, n = case
    w = si.small_workload("dec", hq, hkv, d, cache, dt, n_prompt=n, chunk=n, n_decode=0, seed=hq * 7 + d)
    q, _, _ = si.layer_qkv(w, 0)
    caches = {}
    for layout in ("head_major", "layer_major"):
        caches[layout] = run_appends(kvc, w, layout)
    o = caches["head_major"][1]
    qd = q.cuda()
    for pos in sorted({0, 1, 15, 16, 17, 63, 64, 65, n // 2, n - 2, n - 1}):
        outs = [kvc.decode_attn(caches[l][0], 0, pos, qd[pos]) for l in ("head_major", "layer_major")]
        torch.cuda.synchronize()
        assert torch.equal(outs[0], outs[1]), "layout changed the result at pos %d" % pos
        assert_close(outs[0].cpu().numpy(), o.decode(0, pos, np32(q[pos])), "pos %d" % pos)


def test_decode_long_context_many_splits(kvc):
    w = si.small_workload("long", 40, 8, 128, "q8_0", "bf16", n_prompt=9000, chunk=4096, n_decode=0, seed=5,
                          k_outlier_frac=0.01)
    g, o = run_appends(kvc, w, "layer_major")
    q, _, _ = si.layer_qkv(w, 0)
    for pos in (4095, 8999):
        out = kvc.decode_attn(g, 0, pos, q[pos].cuda())
        assert_close(out.cpu().numpy(), o.decode(0, pos, np32(q[pos])), "pos %d" % pos)


def test_decode_layer_index_and_repeatability(kvc):
    w = si.small_workload("lay", 8, 2, 128, "q8_0", "bf16", n_prompt=500, chunk=500, n_decode=0, seed=9, n_layer=3)
    g, o = run_appends(kvc, w, "head_major")
    q, _, _ = si.layer_qkv(w, 2)
    out1 = kvc.decode_attn(g, 2, 499, q[499].cuda())
    out2 = kvc.decode_attn(g, 2, 499, q[499].cuda())
    assert torch.equal(out1, out2)
    assert_close(out1.cpu().numpy(), o.decode(2, 499, np32(q[499])))
