"""Repeat runs give the same bits.

The same request, run twice on fresh caches and scratch in the bench's launch configuration
(prefill_step per chunk with the item counter and the incremental copy, the decode loop in a CUDA
graph, the state round trip), must give identical outputs, cache bytes and state stream: the
persistent prefill CTAs take their items in whatever order they finish, and each decode step's
splits finish in any order, so a result that depended on timing would show here.
"""

import pytest
import torch

import bench
import seeded_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


def run_request(kvc, w, inputs):
    req = bench.GpuRequest(kvc, w, torch.device("cuda", 0), host_copies=False, inputs=inputs)
    req.step()
    req.capture()
    req.step()
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    return req


@pytest.mark.parametrize("cache,chunk", [("q8_0", 1024), ("f16", 512)])
def test_two_runs_give_the_same_bits(kvc, cache, chunk):
    w = si.small_workload("determ", 40, 8, 128, cache, "bf16", n_prompt=6000, chunk=chunk, n_decode=16, seed=123,
                          k_outlier_frac=0.01)
    inputs = [tuple(t.cuda() for t in si.layer_qkv(w, 0))]
    a = run_request(kvc, w, inputs)
    b = run_request(kvc, w, inputs)
    assert torch.equal(a.out_p, b.out_p)
    assert torch.equal(a.out_d, b.out_d)
    assert torch.equal(a.state, b.state)
    for kv in (0, 1):
        assert torch.equal(a.dst.codes(kv)[0, :w.n_tokens], b.dst.codes(kv)[0, :w.n_tokens])
