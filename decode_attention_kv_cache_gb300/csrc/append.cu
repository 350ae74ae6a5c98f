// Append kernel: quantise a chunk's K/V rows into q8_0 blocks, or round them to
// f16, and store them at their cache positions.
//
// The q8_0 block (32 values along head_dim, fp16 scale d = amax/127, int8
// codes q = round(x/d)) is the one the pages' "q8_0 device-resident cache"
// names (llama.cpp PR #58 "completion : allow the prompt to be processed
// under its own split mode", section "Why"); the f16 cache is the one of
// llama.cpp PR #59 "llama : switch the split mode of a live context",
// section "Why".  The arithmetic repeats, bit for bit, the float32 op order:
// amax exact, d = amax/127 and x/d by IEEE division, ties away from zero,
// fp16 by round to nearest even.
//
// Work split.  q8_0: one thread per 32-value block.  A warp's 32 blocks are
// one contiguous run of input, loaded 16 bytes per lane (consecutive lanes on
// consecutive chunks) into shared memory, from which each lane takes its own
// block; 32 code bytes and one 2-byte scale are stored per block.  The block
// quantiser (quant.cuh) is shared with the fused decode step.  f16: one
// thread per 8 values.  HBM-bound.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "kvc_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace kvc {
namespace {

// Where input token t goes: one cache, token t at position pos0 + t ...
struct OneCache {
    void *kq, *vq;
    uint16_t *ks, *vs;
    Geom g;
    int pos0;
    __device__ __forceinline__ int64_t pos(int t) const { return (int64_t)pos0 + t; }
    __device__ __forceinline__ const Geom &geom(int) const { return g; }
    __device__ __forceinline__ void *codes(bool is_v, int) const { return is_v ? vq : kq; }
    __device__ __forceinline__ uint16_t *scales(bool is_v, int) const { return is_v ? vs : ks; }
};
// ... or one token per sequence: token t into cache t at position pos[t]
constexpr int MAX_SEQ = 8;
struct PerSeqCaches {
    void *kq[MAX_SEQ], *vq[MAX_SEQ];
    uint16_t *ks[MAX_SEQ], *vs[MAX_SEQ];
    Geom g[MAX_SEQ];
    int p[MAX_SEQ];
    __device__ __forceinline__ int64_t pos(int t) const { return p[t]; }
    __device__ __forceinline__ const Geom &geom(int t) const { return g[t]; }
    __device__ __forceinline__ void *codes(bool is_v, int t) const { return is_v ? vq[t] : kq[t]; }
    __device__ __forceinline__ uint16_t *scales(bool is_v, int t) const { return is_v ? vs[t] : ks[t]; }
};

// f16 cache: grid.x covers units of 8 values of one tensor; grid.y selects K (0) or V (1).
template <int DT, class DST>
__global__ void __launch_bounds__(256) append_f16_kernel(
    const void *__restrict__ k, const void *__restrict__ v, int64_t n_units, int units_per_tok,
    int units_per_head, const DST dst_of, int layer) {
    // a kernel launched after this one as a programmatic dependent (the decode split pass) may be
    // scheduled now; it waits for this grid's completion before it reads the cache.  This grid is
    // itself launched as a programmatic dependent: it waits for the kernel before it to complete
    // before it reads its inputs or writes the cache.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool is_v = blockIdx.y != 0;
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= n_units) return;
    const int tok = (int)(u / units_per_tok);
    const int rem = (int)(u % units_per_tok);
    const int head = rem / units_per_head;
    const int c = rem % units_per_head;  // which 8-value group along head_dim
    float x[8];
    load_inputs8<DT>(is_v ? v : k, u * 8, x);
    const int64_t pos = dst_of.pos(tok);
    const Geom &g = dst_of.geom(tok);
    const int64_t code_off = layer * g.c_layer + pos * g.c_tok + head * g.c_head + (int64_t)c * 8;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = ptx::pack_half2(x[2 * i], x[2 * i + 1]);
    uint16_t *dst = static_cast<uint16_t *>(dst_of.codes(is_v, tok)) + code_off;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// the values of one 16-byte input chunk (8 bf16 / f16 or 4 f32) as floats
template <int DT>
__device__ __forceinline__ void chunk_values(const uint4 &u, float *x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (DT == KVC_IN_F32) {
            x[i] = __uint_as_float(w[i]);
        } else if constexpr (DT == KVC_IN_BF16) {
            // bf16 -> f32 is exact: the bf16 bits are the top half of the f32
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            x[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFF)));
            x[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
        }
    }
}

// Staging slot of 16-byte chunk c of a warp's input: XOR-swizzled so that lanes storing consecutive
// chunks and lanes reading their own block's chunks are both free of bank conflicts.
__device__ __forceinline__ int stage_slot(int c) { return c ^ ((c >> 3) & 7); }

// q8_0 cache: one thread per 32-value block; grid.y selects K (0) or V (1).
template <int DT, class DST>
__global__ void __launch_bounds__(256) append_q8_kernel(
    const void *__restrict__ k, const void *__restrict__ v, int64_t n_blocks, int nb, int H, const DST dst_of,
    int layer) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");   // as in append_f16_kernel
    constexpr int ESZ = DT == KVC_IN_F32 ? 4 : 2;
    constexpr int CPB = 2 * ESZ;                   // 16-byte input chunks per block
    __shared__ uint4 stage[8][32 * CPB];
    const bool is_v = blockIdx.y != 0;
    const int lane = threadIdx.x & 31;
    uint4 *S = stage[threadIdx.x >> 5];
    const int64_t blk0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x - lane;   // the warp's first block
    if (blk0 >= n_blocks) return;   // the whole warp
    const int nwc = (int)min((int64_t)32, n_blocks - blk0) * CPB;                 // the warp's input chunks
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(is_v ? v : k) + blk0 * 32 * ESZ);
    {
        uint4 t[CPB];
#pragma unroll
        for (int m = 0; m < CPB; ++m) {
            const int c = 32 * m + lane;
            t[m] = c < nwc ? __ldcg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int m = 0; m < CPB; ++m) S[stage_slot(32 * m + lane)] = t[m];
    }
    __syncwarp();
    const int64_t blk = blk0 + lane;
    if (blk >= n_blocks) return;
    float x[32];
#pragma unroll
    for (int j = 0; j < CPB; ++j) chunk_values<DT>(S[stage_slot(CPB * lane + j)], x + j * (16 / ESZ));
    const int64_t row = blk / nb;                    // (token, head) in input order
    const int b = (int)(blk - row * nb);
    const int tok = (int)(row / H), head = (int)(row - (int64_t)tok * H);
    uint32_t packed[8];
    const uint16_t scale = q8_0_quantize32(x, packed);
    const int64_t pos = dst_of.pos(tok);
    const Geom &g = dst_of.geom(tok);
    int8_t *dst = static_cast<int8_t *>(dst_of.codes(is_v, tok)) + layer * g.c_layer + pos * g.c_tok +
                  head * g.c_head + b * 32;
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    dst_of.scales(is_v, tok)[layer * g.s_layer + pos * g.s_tok + head * g.s_head + b] = scale;
}

// n tokens of k and v ([n][H_kv][head_dim]) to the destinations dst_of gives them; desc: their shape
// Launched as a programmatic dependent of the kernel before it in the stream: its launch overlaps
// that kernel's tail, and the kernel waits on the device (griddepcontrol.wait) before touching memory.
template <int DT, class DST>
cudaError_t launch_t(const kvc_desc &desc, const DST &dst_of, int layer, int n, const void *k, const void *v,
                     cudaStream_t s) {
    const int threads = 256;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (desc.type == KVC_Q8_0) {
        const int nb = desc.head_dim / 32;
        const int64_t n_blocks = (int64_t)n * desc.n_head_kv * nb;
        cfg.gridDim = dim3((unsigned)((n_blocks + threads - 1) / threads), 2);
        return cudaLaunchKernelEx(&cfg, append_q8_kernel<DT, DST>, k, v, n_blocks, nb, (int)desc.n_head_kv, dst_of,
                                  layer);
    } else {
        const int units_per_head = desc.head_dim / 8;
        const int units_per_tok = units_per_head * desc.n_head_kv;
        const int64_t n_units = (int64_t)n * units_per_tok;
        cfg.gridDim = dim3((unsigned)((n_units + threads - 1) / threads), 2);
        return cudaLaunchKernelEx(&cfg, append_f16_kernel<DT, DST>, k, v, n_units, units_per_tok, units_per_head,
                                  dst_of, layer);
    }
}

template <class DST>
int launch_dtype(const kvc_desc &desc, const DST &dst_of, int layer, int n, const void *k, const void *v, int dtype,
                 cudaStream_t s) {
    cudaError_t e;
    switch (dtype) {
        case KVC_IN_F32: e = launch_t<KVC_IN_F32>(desc, dst_of, layer, n, k, v, s); break;
        case KVC_IN_BF16: e = launch_t<KVC_IN_BF16>(desc, dst_of, layer, n, k, v, s); break;
        default: e = launch_t<KVC_IN_F16>(desc, dst_of, layer, n, k, v, s); break;
    }
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? KVC_OK : KVC_ECUDA;
}

}  // namespace

int launch_append(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *k,
                  const void *v, int dtype, cudaStream_t s) {
    if (n_tokens == 0) return KVC_OK;
    OneCache d;
    d.kq = c.k_q;
    d.vq = c.v_q;
    d.ks = static_cast<uint16_t *>(c.k_s);
    d.vs = static_cast<uint16_t *>(c.v_s);
    d.g = geom_of(c.d);
    d.pos0 = pos0;
    return launch_dtype(c.d, d, layer, n_tokens, k, v, dtype, s);
}

int append_max_batch() { return MAX_SEQ; }

int launch_append_batch(const kvc_cache *caches, int n_seq, int layer, const int *pos, const void *k, const void *v,
                        int dtype, cudaStream_t s) {
    PerSeqCaches d;
    memset(&d, 0, sizeof(d));
    for (int i = 0; i < n_seq; ++i) {
        d.kq[i] = caches[i].k_q;
        d.vq[i] = caches[i].v_q;
        d.ks[i] = static_cast<uint16_t *>(caches[i].k_s);
        d.vs[i] = static_cast<uint16_t *>(caches[i].v_s);
        d.g[i] = geom_of(caches[i].d);
        d.p[i] = pos[i];
    }
    return launch_dtype(caches[0].d, d, layer, n_seq, k, v, dtype, s);
}

}  // namespace kvc
