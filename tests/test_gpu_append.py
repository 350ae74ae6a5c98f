"""kv_cache_append on the GPU: cache bytes bit-exact with the oracle."""

import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity_util import assert_cache_equal, np32
from oracle.cache import OracleCache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


def run_appends(kvc, w, layout, layers=None):
    o = OracleCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
    g = kvc.KVCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, layout)
    for layer in (range(w.n_layer) if layers is None else layers):
        _, k, v = si.layer_qkv(w, layer)
        kd, vd = k.cuda(), v.cuda()
        for p, c in w.chunks():
            kvc.kv_cache_append(g, layer, p, kd[p:p + c], vd[p:p + c])
            o.append(layer, p, np32(k[p:p + c]), np32(v[p:p + c]))
        for p in range(w.n_prompt, w.n_tokens):
            kvc.kv_cache_append(g, layer, p, kd[p:p + 1], vd[p:p + 1])
            o.append(layer, p, np32(k[p:p + 1]), np32(v[p:p + 1]))
    torch.cuda.synchronize()
    return g, o


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
@pytest.mark.parametrize("layout", ["head_major", "layer_major"])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16", "f16"])
def test_append_bit_exact(kvc, cache_type, layout, in_dtype):
    w = si.small_workload("a", 8, 4, 128, cache_type, in_dtype, n_prompt=300, chunk=97, n_decode=3, seed=11,
                          n_layer=2, k_outlier_frac=0.02)
    g, o = run_appends(kvc, w, layout)
    assert_cache_equal(g, o, w.n_tokens)


@pytest.mark.parametrize("head_dim,n_head_kv", [(32, 1), (64, 2), (96, 3), (256, 2)])
def test_append_other_shapes(kvc, head_dim, n_head_kv):
    for layout in ("head_major", "layer_major"):
        w = si.small_workload("s", n_head_kv, n_head_kv, head_dim, "q8_0", "bf16", n_prompt=70, chunk=33,
                              n_decode=2, seed=head_dim)
        g, o = run_appends(kvc, w, layout)
        assert_cache_equal(g, o, w.n_tokens)


def test_append_special_blocks(kvc):
    # zero blocks, exact ties, subnormal and large scales, an underflowing scale
    H, D = 2, 64
    x = np.zeros((6, H, D), np.float32)
    x[1, 0, 0] = 15.875
    x[1, 0, 1:9] = [0.0625, -0.0625, 0.1875, -0.1875, 0.3125, -0.3125, 15.8125, -15.8125]
    x[2, 0, :32] = np.float32(127 * 2.0 ** -20) * np.linspace(-1, 1, 32, dtype=np.float32)
    x[2, 1, 32:] = np.float32(3 * 2.0 ** -25) * 127
    x[3, 0, :] = np.linspace(-3000, 3000, D, dtype=np.float32)
    x[4, 1, 5] = np.float32(2.0 ** -144)
    x[5] = np.random.default_rng(0).standard_normal((H, D)).astype(np.float32) * 1e-3
    for cache_type in ("q8_0", "f16"):
        for layout in ("head_major", "layer_major"):
            o = OracleCache(1, 8, H, D, cache_type)
            g = kvc.KVCache(1, 8, H, D, cache_type, layout)
            t = torch.from_numpy(x).cuda()
            kvc.kv_cache_append(g, 0, 1, t, -t)
            o.append(0, 1, x, -x)
            torch.cuda.synchronize()
            # positions 1..6 written; compare them (position 0 untouched on both sides is not compared)
            img = o.device_image(layout)
            for kv in (0, 1):
                gc = g.codes(kv).cpu()
                oc = img[2 * kv]
                sl = (slice(None), slice(None), slice(1, 7)) if layout == "head_major" else (slice(None), slice(1, 7))
                if cache_type == "q8_0":
                    assert np.array_equal(gc[sl].numpy(), oc[sl])
                    assert np.array_equal(g.scales(kv).cpu()[sl].view(torch.int16).numpy(), img[2 * kv + 1][sl].view(np.int16))
                else:
                    assert np.array_equal(gc[sl].view(torch.int16).numpy(), oc[sl].view(np.int16))


def test_append_leaves_other_positions_alone(kvc):
    g = kvc.KVCache(2, 64, 2, 64, "q8_0", "layer_major")
    for kv in (0, 1):
        g.codes(kv).fill_(7)
        g.scales(kv).fill_(1.5)
    k = torch.randn(5, 2, 64, device="cuda")
    kvc.kv_cache_append(g, 1, 10, k, k)
    torch.cuda.synchronize()
    c = g.codes(0).cpu()
    mask = torch.ones_like(c, dtype=torch.bool)
    mask[1, 10:15] = False
    assert (c[mask] == 7).all()
    s = g.scales(1).cpu()
    smask = torch.ones_like(s, dtype=torch.bool)
    smask[1, 10:15] = False
    assert (s[smask] == 1.5).all()
