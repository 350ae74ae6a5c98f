"""Guard bytes around every buffer the path writes.

Each device buffer (the cache's codes and scales, the prefill and decode scratch, the outputs, the
state stream) sits between two 4 KB runs of seeded bytes.  A prompt (append + prefill_chunk_attn,
then prefill_step chunks with the incremental fp16 copy), decode steps up to the cache's last
position, and a state round trip into a second guarded cache must leave every guard byte as it was.
The cache has two layers and the calls use the last one, so the writes reach the ends of the
buffers in both layouts.  This stands in for a memory checker, which is not run on these GPUs.
"""

import ctypes

import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu

G = 4096   # guard bytes on each side; a multiple of 256 keeps the inner buffer's alignment


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


class Guarded:
    """nbytes of device memory between two guards of seeded bytes."""

    def __init__(self, nbytes, seed):
        self.n = max(int(nbytes), 16)
        gen = torch.Generator().manual_seed(seed)
        self.pattern = torch.randint(0, 256, (2 * G,), dtype=torch.uint8, generator=gen)
        self.buf = torch.empty(self.n + 2 * G, dtype=torch.uint8, device="cuda")
        self.buf[:G] = self.pattern[:G].cuda()
        self.buf[G + self.n:] = self.pattern[G:].cuda()
        self.inner = self.buf[G:G + self.n]

    def as_f32(self, shape):
        return self.inner.view(torch.float32)[: int(torch.tensor(shape).prod())].view(shape)

    def intact(self):
        b = self.buf.cpu()
        return torch.equal(b[:G], self.pattern[:G]) and torch.equal(b[G + self.n:], self.pattern[G:])


def guarded_cache(kvc, guards, n_layer, n_ctx, n_head_kv, head_dim, cache, layout, seed):
    """A KVCache whose four buffers are guarded allocations."""
    g = kvc.KVCache(n_layer, n_ctx, n_head_kv, head_dim, cache, layout)
    gb = [Guarded(n, seed + i) for i, n in enumerate(g._sizes)]
    guards.extend(gb)
    g._bufs = [x.inner for x in gb]
    p = [ctypes.c_void_p(x.inner.data_ptr()) for x in gb]
    if cache != "q8_0":
        p[1] = p[3] = ctypes.c_void_p(0)
    assert kvc.lib.kvc_cache_init(ctypes.byref(g.c), ctypes.byref(g.desc), p[0], p[1], p[2], p[3]) == 0
    return g


@pytest.mark.parametrize("cache,layout,d", [("q8_0", "head_major", 128), ("q8_0", "layer_major", 128),
                                            ("f16", "layer_major", 128), ("q8_0", "head_major", 64),
                                            ("f16", "head_major", 64)])
def test_no_write_outside_the_buffers(kvc, cache, layout, d):
    hq, hkv, n_ctx, n_prompt, chunk, layer = 10, 2, 600, 590, 256, 1
    w = si.small_workload("guard", hq, hkv, d, cache, "bf16", n_prompt=n_prompt, chunk=chunk,
                          n_decode=n_ctx - n_prompt, seed=d + len(layout), n_ctx=n_ctx, n_layer=2)
    q, k, v = (t.cuda() for t in si.layer_qkv(w, layer))
    guards = []
    g = guarded_cache(kvc, guards, 2, n_ctx, hkv, d, cache, layout, seed=1)
    pscr = Guarded(g.prefill_scratch_bytes(hq, chunk), 11)
    dscr = Guarded(g.scratch_bytes(hq), 12)
    out_p = Guarded(n_prompt * hq * d * 4, 13)
    out_d = Guarded((n_ctx - n_prompt) * hq * d * 4, 14)
    guards += [pscr, dscr, out_p, out_d]
    op = out_p.as_f32((n_prompt, hq, d))
    od = out_d.as_f32((n_ctx - n_prompt, hq, d))
    for i, (p, c) in enumerate(w.chunks(chunk)):
        if i == 0:
            kvc.kv_cache_append(g, layer, p, k[p:p + c], v[p:p + c])
            kvc.prefill_chunk_attn(g, layer, p, q[p:p + c], out=op[p:p + c], scratch=pscr.inner)
        else:
            kvc.prefill_step(g, layer, p, q[p:p + c], k[p:p + c], v[p:p + c], out=op[p:p + c], scratch=pscr.inner,
                             copy_valid=p)
    for i, p in enumerate(range(n_prompt, n_ctx)):
        kvc.decode_step(g, layer, p, q[p], k[p], v[p], out=od[i], scratch=dscr.inner)
    state = Guarded(g.state_size(n_ctx), 15)
    guards.append(state)
    kvc.kv_state_get(g, n_ctx, dst=state.inner)
    g2 = guarded_cache(kvc, guards, 2, n_ctx, hkv, d, cache, "head_major" if layout == "layer_major" else
                       "layer_major", seed=21)
    assert kvc.kv_state_set(g2, state.inner) == n_ctx
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    assert torch.isfinite(op).all() and torch.isfinite(od).all()
    bad = [i for i, x in enumerate(guards) if not x.intact()]
    assert not bad, "guard bytes changed around buffers %s" % bad
    # the restored cache packs to the same stream
    again = Guarded(g2.state_size(n_ctx), 16)
    kvc.kv_state_get(g2, n_ctx, dst=again.inner)
    torch.cuda.synchronize()
    assert torch.equal(again.inner, state.inner) and again.intact()


def test_guard_check_sees_a_changed_byte(cuda_device):
    # the checker itself: one byte just past the inner buffer, or just before it, changed by a copy
    for where in (G + 1000, G - 1):
        x = Guarded(1000, 3)
        assert x.intact()
        x.buf[where:where + 1] ^= 1
        assert not x.intact()


@pytest.mark.parametrize("cache", ["q8_0", "f16"])
def test_batched_calls_stay_inside(kvc, cache):
    # three sequences of different lengths in guarded caches of both layouts: batched appends and
    # decode steps, the last sequence up to its cache's last position
    hq, hkv, d, n_ctx = 10, 2, 128, 400
    lengths = [390, 120, 7]
    ws = [si.small_workload("gb%d" % i, hq, hkv, d, cache, "bf16", n_prompt=n, chunk=n, n_decode=n_ctx - n,
                            seed=90 + i, n_ctx=n_ctx) for i, n in enumerate(lengths)]
    qkv = [tuple(t.cuda() for t in si.layer_qkv(w, 0)) for w in ws]
    guards = []
    caches = [guarded_cache(kvc, guards, 1, n_ctx, hkv, d, cache, ("head_major", "layer_major")[i % 2], seed=40 + 4 * i)
              for i in range(3)]
    pscr = Guarded(caches[0].prefill_scratch_bytes(hq, max(lengths)), 51)
    guards.append(pscr)
    for g, (q, k, v), n in zip(caches, qkv, lengths):
        kvc.prefill_step(g, 0, 0, q[:n], k[:n], v[:n], scratch=pscr.inner)
    per = caches[0].scratch_bytes(hq)
    bscr = Guarded(3 * per, 52)
    out = Guarded(3 * hq * d * 4, 53)
    guards += [bscr, out]
    o = out.as_f32((3, hq, d))
    for t in range(n_ctx - max(lengths)):
        pos = [n + t for n in lengths]
        qb = torch.stack([q[p] for (q, _, _), p in zip(qkv, pos)])
        kb = torch.stack([k[p] for (_, k, _), p in zip(qkv, pos)])
        vb = torch.stack([v[p] for (_, _, v), p in zip(qkv, pos)])
        if t % 2 == 0:
            kvc.decode_step_batch(caches, 0, pos, qb, kb, vb, out=o, scratch=bscr.inner)
        else:
            kvc.kv_cache_append_batch(caches, 0, pos, kb, vb)
            kvc.decode_attn_batch(caches, 0, pos, qb, out=o, scratch=bscr.inner)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    assert torch.isfinite(o).all()
    bad = [i for i, x in enumerate(guards) if not x.intact()]
    assert not bad, "guard bytes changed around buffers %s" % bad
