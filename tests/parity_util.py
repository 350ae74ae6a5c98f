"""Helpers shared by the GPU parity tests: run a workload's request through the
CUDA path and through the oracle on the same seeded inputs, and compare."""

import numpy as np
import torch

import seeded_inputs as si
from oracle.cache import OracleCache

ATOL, RTOL = 2e-3, 1e-2   # attention outputs: |gpu - ref| <= ATOL + RTOL * |ref|, elementwise


def assert_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), "%s: non-finite output" % what
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = (err / bound).max() if err.size else 0.0
    assert (err <= bound).all(), "%s: max abs err %.3g, max rel err %.3g, worst err/bound %.3g" % (
        what, err.max(), (err / np.maximum(np.abs(ref), 1e-30)).max(), worst)


def np32(t):
    """A CPU float32 numpy copy of a tensor (bf16/f16 widen exactly)."""
    return t.detach().float().cpu().numpy()


def oracle_cache_for(w, layout=None):
    return OracleCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)


def gpu_cache_for(kvc, w, layout="head_major"):
    return kvc.KVCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, layout, device="cuda")


def layout_name(layout):
    return layout


def assert_cache_equal(gcache, ocache, n_tokens, layers=None):
    """Bit-exact comparison of the written positions [0, n_tokens) of a device cache with the oracle."""
    img = ocache.device_image(gcache.layout)
    for kv in (0, 1):
        gc = gcache.codes(kv).cpu()
        oc = img[2 * kv]
        if gcache.layout == "head_major":
            gsl, osl = gc[:, :, :n_tokens], oc[:, :, :n_tokens]
        else:
            gsl, osl = gc[:, :n_tokens], oc[:, :n_tokens]
        if gcache.cache_type == "q8_0":
            assert np.array_equal(gsl.numpy(), osl), "codes differ (kv=%d)" % kv
            gs = gcache.scales(kv).cpu()
            os_ = img[2 * kv + 1]
            gss = gs[:, :, :n_tokens] if gcache.layout == "head_major" else gs[:, :n_tokens]
            oss = os_[:, :, :n_tokens] if gcache.layout == "head_major" else os_[:, :n_tokens]
            assert np.array_equal(gss.view(torch.int16).numpy(), oss.view(np.int16)), "scales differ (kv=%d)" % kv
        else:
            assert np.array_equal(gsl.view(torch.int16).numpy(), osl.view(np.int16)), "values differ (kv=%d)" % kv
