"""The five workloads at full size, run exactly as bench.py times them (its GpuRequest:
same chunking, decode loop in a CUDA graph, state packed from the head-major cache and
restored into a layer-major one), checked against the oracle.

Cache and state bytes are compared bit for bit (whole, or on seeded layer samples for the
64-layer stack); attention outputs on a seeded sample of query rows (each chunk's first
and last row and random rows) and decode steps, which the oracle computes one by one.
"""

import numpy as np
import pytest
import torch

import bench
import seeded_inputs as si
from oracle import state as ostate
from oracle.attention import attend
from oracle.cache import OracleCache
from parity_util import assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


def oracle_layer(w, q, k, v, n_tokens):
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
    o.append(0, 0, np32(k[:n_tokens]), np32(v[:n_tokens]))
    return o


def check_layer(w, req, layer, q, k, v, o, rows, dec_steps, what):
    """Sampled prefill rows and decode steps of one layer, and its cache bytes."""
    slot = req.out_slot(layer)
    kh, vh = o.dequantized(0, w.n_tokens)
    for r0 in range(0, rows.size, 64):
        rr = rows[r0:r0 + 64]
        ref = attend(np32(q[rr]), rr, kh, vh)
        assert_close(req.out_p[slot, rr].cpu().numpy(), ref, "%s prefill rows %s" % (what, rr[:3]))
    for i in dec_steps:
        pos = w.n_prompt + i
        ref = attend(np32(q[pos:pos + 1]), np.array([pos]), kh, vh)[0]
        assert_close(req.out_d[slot, i].cpu().numpy(), ref, "%s decode step %d" % (what, i))


def cache_bytes_equal_oracle(req, o, layer, n_tokens):
    img = o.device_image("head_major")
    for kv in (0, 1):
        g = req.src.codes(kv)[:, layer, :n_tokens].cpu()
        ref = img[2 * kv][:, 0, :n_tokens]
        if req.src.cache_type == "q8_0":
            assert np.array_equal(g.numpy(), ref)
            assert np.array_equal(req.src.scales(kv)[:, layer, :n_tokens].cpu().view(torch.int16).numpy(),
                                  img[2 * kv + 1][:, 0, :n_tokens].view(np.int16))
        else:
            assert np.array_equal(g.view(torch.int16).numpy(), ref.view(np.int16))


@pytest.mark.parametrize("name", ["toy_q8_0", "f16_17k", "q8_0_58k"])
def test_single_layer_request(kvc, name):
    w = si.WORKLOADS[name]
    req = bench.GpuRequest(kvc, w, torch.device("cuda", 0), host_copies=False)
    req.step()
    if w.n_decode:
        req.capture()       # the bench replays the decode loop from a graph
        req.step()
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    q, k, v = si.layer_qkv(w, 0)
    o = oracle_layer(w, q, k, v, w.n_tokens)
    cache_bytes_equal_oracle(req, o, 0, w.n_tokens)
    full = name == "toy_q8_0"
    rows = np.arange(w.n_prompt) if full else si.sample_rows(w.seed, w.chunks())
    dec = range(w.n_decode) if full else sorted({0, 1, w.n_decode // 2, w.n_decode - 1})
    check_layer(w, req, 0, q, k, v, o, rows, dec, name)
    # the state: bit-exact with the oracle, and the restored layer-major cache packs to the same bytes
    blob = req.state.cpu().numpy()
    assert np.array_equal(blob, ostate.pack(o, w.n_tokens))
    assert torch.equal(kvc.kv_state_get(req.dst, w.n_tokens), req.state)


def test_chunk_sweep(kvc):
    w = si.WORKLOADS["q8_0_sweep_10k"]
    q, k, v = si.layer_qkv(w, 0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs, states = {}, {}
    for chunk in w.chunk_sweep:
        ww = si.Workload(**{**w.__dict__, "chunk": chunk})
        req = bench.GpuRequest(kvc, ww, torch.device("cuda", 0), host_copies=False, inputs=[(qd, kd, vd)])
        req.step()
        torch.cuda.synchronize()
        outs[chunk] = req.out_p[0].clone()
        states[chunk] = req.state.clone()
    ref_chunk = w.chunk_sweep[0]
    for chunk in w.chunk_sweep[1:]:
        assert torch.equal(outs[chunk], outs[ref_chunk]), "chunk %d output differs from chunk %d" % (chunk, ref_chunk)
        assert torch.equal(states[chunk], states[ref_chunk])
    o = oracle_layer(w, q, k, v, w.n_prompt)
    assert np.array_equal(states[ref_chunk].cpu().numpy(), ostate.pack(o, w.n_prompt))
    rows = si.sample_rows(w.seed, w.chunks(256))
    kh, vh = o.dequantized(0, w.n_prompt)
    for r0 in range(0, rows.size, 64):
        rr = rows[r0:r0 + 64]
        assert_close(outs[ref_chunk][rr].cpu().numpy(), attend(np32(q[rr]), rr, kh, vh), "sweep rows")


def test_layer_stack_state_restore_and_resumed_decode(kvc):
    w = si.WORKLOADS["q8_0_stack64"]
    extra = 4                                   # rows drawn past the request for the resumed decode
    req = bench.GpuRequest(kvc, w, torch.device("cuda", 0), host_copies=False, extra_rows=extra)
    sampled = (0, 1, 31, 63)
    saved = {}

    def keep(layer):
        if layer in sampled:
            saved[layer] = (req.out_p[0].clone(), req.out_d[0].clone())

    req.step(on_layer=keep)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    # restored layer-major cache == original head-major cache, position by position
    n = w.n_tokens
    for kv in (0, 1):
        assert torch.equal(req.dst.codes(kv)[:, :n].permute(2, 0, 1, 3), req.src.codes(kv)[:, :, :n])
        assert torch.equal(req.dst.scales(kv)[:, :n].permute(2, 0, 1, 3), req.src.scales(kv)[:, :, :n])
    rec = ostate.record_bytes(w.n_head_kv, w.head_dim, w.cache)
    blob = req.state
    for layer in sampled:
        q, k, v = (t.cpu() for t in req.dev_in[layer])
        o = oracle_layer(w, q, k, v, n)
        # this layer's records in the stream
        lo = ostate.HEADER_BYTES + layer * n * 2 * rec
        mine = blob[lo:lo + n * 2 * rec].cpu().numpy()
        assert np.array_equal(mine, ostate.pack(o, n)[ostate.HEADER_BYTES:])
        req.out_p[0].copy_(saved[layer][0])
        req.out_d[0].copy_(saved[layer][1])
        rows = si.sample_rows(w.seed + layer, w.chunks(), n_random=2)
        check_layer(w, req, layer, q, k, v, o, rows, (0, w.n_decode - 1), "layer %d" % layer)
        # decode resumes on both caches - the head-major one by decode_step, the restored layer-major
        # one by append + decode_attn: bitwise equal, and equal to the oracle
        qd, kd, vd = req.dev_in[layer]
        for pos in range(n, n + extra):
            outs = [kvc.decode_step(req.src, layer, pos, qd[pos], kd[pos], vd[pos])]
            kvc.kv_cache_append(req.dst, layer, pos, kd[pos:pos + 1], vd[pos:pos + 1])
            outs.append(kvc.decode_attn(req.dst, layer, pos, qd[pos]))
            assert torch.equal(outs[0], outs[1])
        o.append(0, n, np32(k[n:n + extra]), np32(v[n:n + extra]))
        assert_close(outs[0].cpu().numpy(), o.decode(0, n + extra - 1, np32(q[n + extra - 1])), "resumed decode")
