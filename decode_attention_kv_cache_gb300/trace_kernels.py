"""Clock-stamp timelines of one CTA of the decode split pass or the prefill attention pass
(diagnostic; needs a GPU and nvcc).

    python -m decode_attention_kv_cache_gb300.trace_kernels [decode | prefill]

Builds libkvc_trace.so (the library compiled with -DKVC_TRACE, whose
tensor-core passes record clock64 stamps of their pipeline events in one CTA).

decode: fills one layer of 40 query / 8 kv heads at head_dim 128 with
seeded N(0,1) bf16 keys and values (a q8_0 cache of 58,556 tokens, then an
f16 cache of 17,183 tokens), runs decode_attn at the last position three times,
flushes L2, runs it once more and prints that call's timeline in SM cycles
from the CTA's entry:

    per tile   K and V copies issued, S issued (start / end), PV issued (start /
               end), S seen by the softmax, S released, P published, and for
               q8_0 the codes landed and the dequantised tile ready (K and V)
    overall    set-up done, Q' built, first S issue allowed, epilogue start,
               rows stored, merge done, end

plus the median cycles between consecutive S issues.

prefill: fills a q8_0 layer (40 / 8 heads, head_dim 128) with 53,248 seeded
tokens, runs prefill_chunk_attn for the 2,048 rows at position 51,200 with the
full scratch (the attention pass runs over the dequantised fp16 copy) twice,
flushes L2, runs it once more and prints CTA 0's timeline per key tile (in SM
cycles from its first stamp): S allowed (the softmax has read the previous S),
K ready, S issued, P ready seen by the MMA thread, PV issued, and per softmax
warpgroup S seen and P published (warpgroup 0 also S released and the row
maximum exchanged), plus the stage loads of the producer.
"""

import ctypes
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import decode_attention_kv_cache_gb300 as kvc  # noqa: E402
from decode_attention_kv_cache_gb300 import build  # noqa: E402

COLS = ["K copy", "V copy", "S issue", "S issued", "PV issue", "PV issued", "S seen", "S freed", "P ready",
        "K codes", "K ready", "V codes", "V ready"]


def run(lib, cache_type, n_keys, n_ctx):
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    H, Hq, D = 8, 40, 128
    cache = kvc.KVCache(1, n_ctx, H, D, cache_type, "head_major")
    k = torch.randn(n_keys, H, D, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(n_keys, H, D, device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn(Hq, D, device="cuda", generator=g).to(torch.bfloat16)
    kvc.kv_cache_append(cache, 0, 0, k, v)
    scratch = torch.empty(cache.scratch_bytes(Hq), dtype=torch.uint8, device="cuda")
    out = torch.empty(Hq, D, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        kvc.decode_attn(cache, 0, n_keys - 1, q, out=out, scratch=scratch)
    flush.add_(1)
    torch.cuda.synchronize()
    assert lib.kvc_trace_clear() == 0
    kvc.decode_attn(cache, 0, n_keys - 1, q, out=out, scratch=scratch)
    torch.cuda.synchronize()
    buf = np.zeros((16, 64), dtype=np.uint64)
    assert lib.kvc_trace_read(buf.ctypes.data_as(ctypes.c_void_p)) == 0
    t0 = int(buf[0, 0])
    rel = lambda x: (int(x) - t0) if x else -1
    print("== %s cache, %d keys, CTA (split 0, kv head 0)" % (cache_type, n_keys))
    print("set-up done %d, Q' built %d, first S allowed %d, epilogue %d, rows stored %d, merged %d, end %d" % (
        rel(buf[0, 1]), rel(buf[0, 6]), rel(buf[0, 2]), rel(buf[0, 3]), rel(buf[0, 7]), rel(buf[0, 4]),
        rel(buf[0, 5])))
    ntiles = int((buf[3] != 0).sum())
    print("tile " + " ".join("%9s" % c for c in COLS))
    for t in range(ntiles):
        print("%4d " % t + " ".join("%9d" % rel(buf[e, t]) for e in range(1, 14)))
    s_issue = buf[3, :ntiles].astype(np.int64)
    if ntiles > 2:
        print("median cycles between S issues: %d" % int(np.median(np.diff(s_issue))))


PCOLS = ["S allowed", "K ready", "S issued", "P seen", "PV issued", "wg0 S seen", "wg0 S free", "wg0 max",
         "wg0 P", "wg1 S seen", "wg1 P"]


def run_prefill(lib):
    g = torch.Generator(device="cuda")
    g.manual_seed(4321)
    H, Hq, D, n_ctx = 8, 40, 128, 65536
    pos0, C = 51200, 2048
    cache = kvc.KVCache(1, n_ctx, H, D, "q8_0", "head_major")
    k = torch.randn(pos0 + C, H, D, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(pos0 + C, H, D, device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn(C, Hq, D, device="cuda", generator=g).to(torch.bfloat16)
    kvc.kv_cache_append(cache, 0, 0, k, v)
    scratch = cache.prefill_scratch(Hq, C)
    out = torch.empty(C, Hq, D, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        kvc.prefill_chunk_attn(cache, 0, pos0, q, out=out, scratch=scratch)
    flush.add_(1)
    torch.cuda.synchronize()
    assert lib.kvc_ptrace_clear() == 0
    kvc.prefill_chunk_attn(cache, 0, pos0, q, out=out, scratch=scratch)
    torch.cuda.synchronize()
    buf = np.zeros((16, 128), dtype=np.uint64)
    assert lib.kvc_ptrace_read(buf.ctypes.data_as(ctypes.c_void_p)) == 0
    nz = buf[buf != 0]
    t0 = int(nz.min()) if nz.size else 0
    rel = lambda x: (int(x) - t0) if x else -1
    ntiles = int((buf[3] != 0).sum())
    print("== prefill, q8_0 cache over its fp16 copy, 2,048 rows at position 51,200, CTA 0: %d key tiles" % ntiles)
    print("tile " + " ".join("%10s" % c for c in PCOLS))
    for t in range(ntiles):
        print("%4d " % t + " ".join("%10d" % rel(buf[e, t]) for e in range(1, 12)))
    s_iss = buf[3, :ntiles].astype(np.int64)
    if ntiles > 2:
        print("median cycles between S issues: %d" % int(np.median(np.diff(s_iss))))
    nst = int((buf[12] != 0).sum())
    print("producer stage loads issued (first 16): " + " ".join(str(rel(x)) for x in buf[12, :min(nst, 16)]))


def main():
    path = build.build(verbose=True, trace=True)
    kvc.LIB_PATH = path
    lib = ctypes.CDLL(path)
    for f in ("kvc_trace_clear", "kvc_trace_read", "kvc_ptrace_clear", "kvc_ptrace_read"):
        getattr(lib, f).restype = ctypes.c_int
    lib.kvc_trace_read.argtypes = [ctypes.c_void_p]
    lib.kvc_ptrace_read.argtypes = [ctypes.c_void_p]
    what = sys.argv[1] if len(sys.argv) > 1 else "decode"
    if what == "decode":
        run(lib, "q8_0", 58556, 65536)
        run(lib, "f16", 17183, 20480)
    elif what == "prefill":
        run_prefill(lib)
    else:
        raise SystemExit("usage: python -m decode_attention_kv_cache_gb300.trace_kernels [decode | prefill]")


if __name__ == "__main__":
    main()
