// Prefill attention for one chunk of query rows over the KV cache, on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes: for each query row t of the chunk [pos0, pos0 + C) and
// query head h, softmax over keys j <= t of q.khat_j / sqrt(D), applied to
// vhat_j, with kv head h / G (grouped-query attention) - the flash attention
// the pages run over the cache while a prompt is processed in ubatches
// (llama.cpp PR #17 "--split-overlap", section "Results": "native FA";
// llama.cpp PR #58 "completion : allow the prompt to be processed under its
// own split mode", section "Why").
//
// Work decomposition.  A unit is 128 query rows of one query head.  Keys are
// taken in tiles of 256 and cut at ABSOLUTE split boundaries of ST tiles (ST
// is fixed by the cache size): an item is (unit, split).  Persistent CTAs (one
// per SM) take items in split-major, kv-group-major order, so that the CTAs
// running at one time read the same K/V tiles: round-robin, or (prefill_step)
// the next item in that order whenever a CTA is free, from a counter in the
// scratch that the step's first kernel zeroes.  An item whose unit has
// one split writes the output directly; otherwise it writes its partial (O,
// running max, sum), and a second, fully parallel kernel merges each row's
// partials in split order.  Because tiles and splits sit at absolute
// positions and every merge runs in split order, a row's result does not
// depend on how the prompt is cut into chunks.
//
// Tensor memory (512 columns): S = Q K^T of one key tile (256 fp32 columns),
// P = softmax numerators as fp16 (128 columns), O (D columns).  S, P and O
// are separate, so S of the next tile is computed while the softmax of this
// one runs, and the MMA issue order per tile is S(k+1), PV(k).  Both are
// M=128 MMAs; S has N=256.  (Issued back to back without waits, a tile of
// N=256 S and N=128 PV takes the tensor core 4,100 cycles and one with S as
// two N=128 halves 2,440, but here S and PV are issued one barrier apart,
// the split S finishes later, and the kernel measured 5% slower with it.)
//
// One CTA:
//   warp 0      TMA producer: the Q tile of an item, then K and V tiles in
//               the MMA's order K(k0), K(k0+1), V(k0), K(k0+2), V(k0+1), ...
//               (int8 codes into a raw ring for q8_0; fp16 values straight into
//               the operand ring for f16).
//   warp 1      allocates the 512 TMEM columns; one lane issues tcgen05.mma.
//   warps 2-3   put the Q tile in fp16 (bf16 converted in place, f32 read from
//               global memory); Q is released after the item's last S MMA, so
//               the next item's Q loads during this one's tail.
//   warps 4-11  softmax: two warpgroups, each owns 128 of the tile's 256 key
//               columns for all 128 rows (thread = TMEM lane = row).  The two
//               threads of a row exchange their half-row maxima (and at the
//               end the sums) through flagged shared-memory words, so both use
//               the same running max; each group writes its half of P and
//               rescales its half of O (only when the running max grows by
//               more than 2^8).  After an item's last tile they read O out of
//               TMEM and write O / l, or the partial, 32 bytes per store.
//   warps 12-15 (q8_0) dequantise int8 rows into fp16 d*q in the 128-byte
//               swizzled operand layout.
// Every mbarrier wait is bounded (2 s); a wait that gives up sets the device
// status word and the CTA skips its remaining work, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kvc_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace kvc {

__device__ int g_device_status;

namespace {

// Diagnostic build (-DKVC_TRACE, see build.py): CTA 0 of the attention pass records clock64 stamps of its
// pipeline events, event e of its n-th key tile in g_ptrace[e][n], for kvc_ptrace_read.  The stamps change
// no work; a normal build compiles them away.
#ifdef KVC_TRACE
__device__ unsigned long long g_ptrace[16][128];
#define KVC_PTR(ev, n)                                                           \
    do {                                                                       \
        if (blockIdx.x == 0 && (n) < 128) g_ptrace[ev][n] = clock64();          \
    } while (0)
#else
#define KVC_PTR(ev, n) do { } while (0)
#endif

using namespace ptx;

constexpr int BM = 128;           // query rows per unit
constexpr int BN = 256;           // keys per tile
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_P = 256, COL_O = 384;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int MAX_SPLITS = 64;
constexpr int MAX_DYN_SMEM = 232448;   // 227 KB per CTA
// a partial row: D values, the running max, the sum, six pad floats (keeps rows 32-byte aligned)
#define PART_ROW(D) ((D) + 8)

template <int D, bool Q8>
struct Cfg {
    static constexpr int QT_BYTES = BM * D * 2;    // the fp16 Q tile
    static constexpr int ST_BYTES = BN * D * 2;    // one ring stage: a fp16 K or V tile
    static constexpr int RAW_BYTES = BN * D;       // one int8 K or V tile
    static constexpr int NS = Q8 ? (D == 128 ? 2 : 4) : (D == 128 ? 3 : 6);  // fp16 operand ring stages
    static constexpr int NR = Q8 ? (D == 128 ? 2 : 4) : 1;                   // int8 raw ring stages
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = OFF_Q + QT_BYTES;
    static constexpr int OFF_RAW = OFF_RING + NS * ST_BYTES;
    static constexpr int OFF_BAR = OFF_RAW + (Q8 ? NR * RAW_BYTES : 0);
    static constexpr int OFF_RED = OFF_BAR + 384;             // mailbox words [slot][group][row]
    static constexpr int USED = OFF_RED + 2 * 2 * BM * 4;
    static constexpr int ALLOC = (USED + 1024 <= MAX_DYN_SMEM) ? USED + 1024 : MAX_DYN_SMEM;
    static_assert(USED <= MAX_DYN_SMEM, "shared memory plan too large");
    static constexpr int THREADS = Q8 ? 512 : 384;
    // registers per thread: at launch (65536 / THREADS, multiple of 8), then per warpgroup after
    // setmaxnreg; sum over warpgroups of 128 * regs must not exceed THREADS * LAUNCH_REGS
    static constexpr int LAUNCH_REGS = Q8 ? 128 : 168;
    static constexpr int WG0_REGS = Q8 ? 72 : 152;          // producer, MMA issuer, Q warps
    static constexpr int DQ_REGS = 88;                      // dequantising warpgroup (q8_0)
    static constexpr int SM_REGS = 176;                     // each softmax warpgroup
    static_assert(128 * WG0_REGS + 256 * SM_REGS + (Q8 ? 128 * DQ_REGS : 0) <= THREADS * LAUNCH_REGS,
                  "register split exceeds the launch allocation");
    static_assert(NS <= 6 && NR <= 4, "more ring stages than barriers");
    // warps that read each item index: the MMA issuer, the two Q warps, eight softmax warps, (q8_0) four
    // dequantising warps
    static constexpr int ITEM_READERS = Q8 ? 15 : 11;
};

constexpr int NIT = 4;            // slots of the item ring (item indices from the producer to the other roles)
enum Bar {
    B_QFULL, B_QREADY, B_QEMPTY, B_SFULL, B_SFREE, B_PFULL, B_ODONE, B_DRAIN, B_STALL,
    B_RING_FULL, B_RING_EMPTY = B_RING_FULL + 6, B_RAW_FULL = B_RING_EMPTY + 6,
    B_RAW_EMPTY = B_RAW_FULL + 4, B_ITEM_FULL = B_RAW_EMPTY + 4, B_ITEM_EMPTY = B_ITEM_FULL + NIT,
    NBAR = B_ITEM_EMPTY + NIT
};

struct Args {
    const float *q_f32;
    const uint16_t *ks;
    const uint16_t *vs;
    float *out;
    float *part;      // partials [q-tile][head][split][row][PART_ROW]
    unsigned *item_counter;  // null: CTA b takes items b, b + grid, ...; else items come from this counter,
                             // which the kernel before this one on the stream set to zero
    Geom g;
    int layer, pos0, C, kv_len, H_q, G, H_kv, n_qt, ST, smax, n_items;
    int v8;                    // out and part are 32-byte aligned: rows are stored 32 bytes at a time
    float scale_log2;
    uint64_t stall_ns;         // test hook: > 0 makes the MMA thread's first P wait one that runs out
    int cum[MAX_SPLITS + 1];   // items before split index s
    int qtmin[MAX_SPLITS];     // first q-tile whose keys reach split s
};

struct Item {
    int g, h, qt, s, ns, k0, k1, tf, tl;
};

// last absolute position of q-tile qt
__device__ __forceinline__ int unit_tl(const Args &a, int qt) {
    return a.pos0 + min(qt * BM + BM, a.C) - 1;
}

// Items are ordered by split, then kv group, then q-tile (last first: the later q-tiles reach further
// into the split, so the shorter items come last in each group), then head within the group.
__device__ __forceinline__ Item decode_item(const Args &a, int i) {
    Item it;
    int s = 0;
    while (s + 1 < a.smax && a.cum[s + 1] <= i) ++s;
    const int r = i - a.cum[s];
    const int per_g = (a.n_qt - a.qtmin[s]) * a.G;
    it.g = r / per_g;
    const int rem = r - it.g * per_g;
    it.qt = a.n_qt - 1 - rem / a.G;
    it.h = it.g * a.G + rem % a.G;
    it.s = s;
    it.tf = a.pos0 + it.qt * BM;
    it.tl = unit_tl(a, it.qt);
    const int T = it.tl / BN + 1;
    it.ns = (T + a.ST - 1) / a.ST;
    it.k0 = s * a.ST;
    it.k1 = min(T, (s + 1) * a.ST);
    return it;
}

__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4));
}
__device__ __forceinline__ uint32_t sw64(int row, int c) {
    return (uint32_t)(row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
}
// Chunk `cc` (8 halves) of row `row` of an fp16 operand tile of `rows` rows
// (64-half column blocks of rows*128 bytes, 128-byte swizzle inside).
__device__ __forceinline__ uint32_t op_off(int rows, int row, int cc) {
    return (uint32_t)((cc >> 3) * rows * 128) + sw128(row, cc & 7);
}


// 4 int8 codes times the fp16 scale, as two fp16x2 words (one rounding each).  Flipping the sign
// bit makes each code q + 128 as an unsigned byte; under the high byte 0x64 that is the fp16 value
// 1024 + q + 128, exact, and subtracting 1152 leaves q.
__device__ __forceinline__ void dequant4(uint32_t w, __half2 d2, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 ra = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&a), bias), d2);
    __half2 rb = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&b), bias), d2);
    lo = *reinterpret_cast<uint32_t *>(&ra);
    hi = *reinterpret_cast<uint32_t *>(&rb);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// One row's split partials merged: out = sum_s w_s O_s / sum_s w_s l_s, w_s = 2^(m_s - max_s m_s), the
// splits taken in split order; the four output values at columns c4 .. c4 + 3 of the row whose split-0
// partial starts at `base` (split s at base + s * sstride).
template <int D>
__device__ __forceinline__ float4 merge_row4(const float *base, int64_t sstride, int ns, int c4) {
    float M = -INFINITY, Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float ms, float ls, float4 v) {
        const float w = (ms == -INFINITY) ? 0.f : (ms == M ? 1.f : ex2(ms - M));
        Lsum = fmaf(w, ls, Lsum);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    };
    constexpr int MS = 8;   // up to MS splits: every load is issued before the first use (one round trip)
    if (ns <= MS) {
        float2 ml[MS];
        float4 v[MS];
#pragma unroll
        for (int s = 0; s < MS; ++s) {
            ml[s] = make_float2(-INFINITY, 0.f);
            v[s] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s < ns) {
                ml[s] = __ldcg(reinterpret_cast<const float2 *>(base + s * sstride + D));
                v[s] = __ldcg(reinterpret_cast<const float4 *>(base + s * sstride + c4));
            }
        }
#pragma unroll
        for (int s = 0; s < MS; ++s)
            if (s < ns) M = fmaxf(M, ml[s].x);
#pragma unroll
        for (int s = 0; s < MS; ++s)
            if (s < ns) add(ml[s].x, ml[s].y, v[s]);
    } else {
#pragma unroll 4
        for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(base + s * sstride + D));
#pragma unroll 4
        for (int s = 0; s < ns; ++s) {
            const float *ps = base + s * sstride;
            add(__ldcg(ps + D), __ldcg(ps + D + 1), __ldcg(reinterpret_cast<const float4 *>(ps + c4)));
        }
    }
    const float inv_l = 1.f / Lsum;
    return make_float4(acc.x * inv_l, acc.y * inv_l, acc.z * inv_l, acc.w * inv_l);
}

template <int D, bool Q8, int QDT>
__global__ void __launch_bounds__(Cfg<D, Q8>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Args a) {
    using L = Cfg<D, Q8>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    if (sm + L::USED > smem_raw + L::ALLOC) {  // the operand tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(&g_device_status, 2);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + NBAR);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    volatile int *s_item = reinterpret_cast<volatile int *>(s_tmem + 2);
    volatile uint32_t *s_mb = reinterpret_cast<volatile uint32_t *>(sm + L::OFF_RED);
    static_assert(NBAR * 8 + 8 + 4 * NIT <= 384, "barrier area too small");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        *s_abort = 0;
        mbar_init(&bars[B_QFULL], 1);
        mbar_init(&bars[B_QREADY], 64);
        mbar_init(&bars[B_QEMPTY], 1);
        mbar_init(&bars[B_SFULL], 1);
        mbar_init(&bars[B_SFREE], 256);
        mbar_init(&bars[B_PFULL], 256);
        mbar_init(&bars[B_ODONE], 1);
        // mailbox words start with flag bit 1: the first value written to each slot carries flag 0
        for (int i = 0; i < 2 * 2 * BM; ++i) reinterpret_cast<uint32_t *>(sm + L::OFF_RED)[i] = 1u;
        mbar_init(&bars[B_DRAIN], 1);
        mbar_init(&bars[B_STALL], 1);   // nothing arrives here: only the test hook waits on it
        for (int s = 0; s < L::NS; ++s) {
            mbar_init(&bars[B_RING_FULL + s], Q8 ? 128 : 1);
            mbar_init(&bars[B_RING_EMPTY + s], 1);
        }
        for (int s = 0; s < L::NR; ++s) {
            mbar_init(&bars[B_RAW_FULL + s], 1);
            mbar_init(&bars[B_RAW_EMPTY + s], 128);
        }
        for (int s = 0; s < NIT; ++s) {
            mbar_init(&bars[B_ITEM_FULL + s], 1);
            mbar_init(&bars[B_ITEM_EMPTY + s], L::ITEM_READERS);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int first_item = blockIdx.x, stride = gridDim.x;
    // The CTA's items, in order: the producer takes each index (the next value of the item counter, or
    // the next of blockIdx.x + n * gridDim.x) and passes it through a ring of NIT slots; every other role
    // reads the same sequence.  An index of n_items ends it.  A reader frees its slot as soon as it has
    // read the index, so the producer is never held by a role that waits for the producer's earlier data.
    auto take_item = [&](uint32_t &seq, bool whole_warp) -> int {
        const int slot = seq % NIT;
        if (!mbar_wait(&bars[B_ITEM_FULL + slot], (seq / NIT) & 1, s_abort)) return -1;
        const int i = s_item[slot];
        ++seq;
        if (whole_warp) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(&bars[B_ITEM_EMPTY + slot]);
        } else {
            mbar_arrive(&bars[B_ITEM_EMPTY + slot]);
        }
        return i;
    };
    // launched as a programmatic dependent of the kernel before it on the stream (normally the append
    // of this chunk's keys): the set-up above overlapped that kernel's tail, and everything global
    // (the cache, Q, the outputs) is read and written only past this wait.  The merge pass may be
    // scheduled from now on; it waits for this grid in turn.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp < 4) setmaxnreg_dec<L::WG0_REGS>();  // producer, MMA issuer and the Q warps
    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t ring_seq = 0, raw_seq = 0, q_seq = 0;
            bool ok = true;
            // the next K or V tile of kv group g into the raw (q8_0) or operand (f16) ring
            auto load_kv = [&](int kv, int k, int g) -> bool {
                const CUtensorMap *m = kv ? &tm_v : &tm_k;
                if (Q8) {
                    const int rs = raw_seq % L::NR;
                    if (raw_seq >= (uint32_t)L::NR &&
                        !mbar_wait(&bars[B_RAW_EMPTY + rs], ((raw_seq / L::NR) - 1) & 1, s_abort))
                        return false;
                    mbar_arrive_expect_tx(&bars[B_RAW_FULL + rs], L::RAW_BYTES);
                    tma_load_3d(sm + L::OFF_RAW + rs * L::RAW_BYTES, m, &bars[B_RAW_FULL + rs], 0, k * BN, g);
                    ++raw_seq;
                } else {
                    const int st = ring_seq % L::NS;
                    if (ring_seq >= (uint32_t)L::NS &&
                        !mbar_wait(&bars[B_RING_EMPTY + st], ((ring_seq / L::NS) - 1) & 1, s_abort))
                        return false;
                    KVC_PTR(12, ring_seq);
                    mbar_arrive_expect_tx(&bars[B_RING_FULL + st], L::ST_BYTES);
                    for (int dh = 0; dh < D / 64; ++dh)
                        tma_load_3d(sm + L::OFF_RING + st * L::ST_BYTES + dh * BN * 128, m, &bars[B_RING_FULL + st],
                                    dh * 64, k * BN, g);
                    ++ring_seq;
                }
                return true;
            };
            for (uint32_t item_seq = 0; ok; ++item_seq) {
                const int slot = item_seq % NIT;
                if (item_seq >= NIT &&
                    !mbar_wait(&bars[B_ITEM_EMPTY + slot], ((item_seq / NIT) - 1) & 1, s_abort))
                    break;
                int i = a.item_counter ? (int)atomicAdd(a.item_counter, 1u) : first_item + (int)item_seq * stride;
                if (i > a.n_items) i = a.n_items;
                s_item[slot] = i;
                mbar_arrive(&bars[B_ITEM_FULL + slot]);
                if (i == a.n_items) break;
                const Item it = decode_item(a, i);
                if (q_seq > 0 && !mbar_wait(&bars[B_QEMPTY], (q_seq - 1) & 1, s_abort)) break;
                if (QDT != KVC_IN_F32) {
                    mbar_arrive_expect_tx(&bars[B_QFULL], L::QT_BYTES);
                    for (int dh = 0; dh < D / 64; ++dh)
                        tma_load_3d(sm + L::OFF_Q + dh * BM * 128, &tm_q, &bars[B_QFULL], dh * 64, it.h, it.qt * BM);
                } else {
                    mbar_arrive(&bars[B_QFULL]);  // the Q warps load f32 Q themselves
                }
                ++q_seq;
                ok = load_kv(0, it.k0, it.g);
                for (int k = it.k0; ok && k < it.k1; ++k) {
                    if (k + 1 < it.k1) ok = load_kv(0, k + 1, it.g);
                    if (ok) ok = load_kv(1, k, it.g);
                }
            }
            if (*s_abort) {
                // after a wait gave up: let the copies still in flight land before the CTA exits
                volatile int never = 0;
                const uint32_t n = Q8 ? raw_seq : ring_seq, stages = Q8 ? L::NR : L::NS;
                for (uint32_t st = 0; st < stages && st < n; ++st) {
                    const uint32_t last = st + ((n - 1 - st) / stages) * stages;
                    mbar_wait(&bars[(Q8 ? B_RAW_FULL : B_RING_FULL) + st], (last / stages) & 1, &never, 200000000ull);
                }
                if (QDT != KVC_IN_F32 && q_seq > 0) mbar_wait(&bars[B_QFULL], (q_seq - 1) & 1, &never, 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(BM, BN, 0, 0);
            constexpr uint32_t IDESC_O = idesc_f16(BM, D, 0, 1);
            const uint32_t sQ = smem_u32(sm + L::OFF_Q), sRing = smem_u32(sm + L::OFF_RING);
            uint32_t ring_seq = 0, q_seq = 0, s_issued = 0, p_seq = 0;
            bool ok = true;
            auto ring_wait = [&](uint32_t seq) -> bool {
                if (!mbar_wait(&bars[B_RING_FULL + seq % L::NS], (seq / L::NS) & 1, s_abort)) return false;
                tc_fence_after();
                return true;
            };
            // S = Q K^T of the next K tile in the ring.  It overwrites the previous S, which the
            // softmax must have read out (s_free).
            auto issue_s = [&]() -> bool {
                if (s_issued > 0 && !mbar_wait(&bars[B_SFREE], (s_issued - 1) & 1, s_abort)) return false;
                KVC_PTR(1, s_issued);
                const uint32_t seq = ring_seq++;
                if (!ring_wait(seq)) return false;
                KVC_PTR(2, s_issued);
                const uint32_t kb = sRing + (seq % L::NS) * L::ST_BYTES;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t kk = (ks & 3) * 32;
                    umma_f16_ss(tmem + COL_S, sdesc_sw128(sQ + (ks >> 2) * (BM * 128) + kk, 16, 1024),
                                sdesc_sw128(kb + (ks >> 2) * (BN * 128) + kk, 16, 1024), IDESC_S, ks > 0);
                }
                umma_commit(&bars[B_SFULL]);
                umma_commit(&bars[B_RING_EMPTY + seq % L::NS]);
                KVC_PTR(3, s_issued);
                ++s_issued;
                return true;
            };
            // O (+)= P V: P fp16 from TMEM, V MN-major in the ring stage
            auto issue_pv = [&](bool acc) -> bool {
                const uint32_t seq = ring_seq++;
                KVC_PTR(4, p_seq - 1);
                if (!ring_wait(seq)) return false;
                const uint32_t vb = sRing + (seq % L::NS) * L::ST_BYTES;
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                    umma_f16_ts(tmem + COL_O, tmem + COL_P + ks * 8, sdesc_sw128(vb + ks * 16 * 128, BN * 128, 1024),
                                IDESC_O, (acc || ks > 0) ? 1u : 0u);
                umma_commit(&bars[B_ODONE]);
                umma_commit(&bars[B_RING_EMPTY + seq % L::NS]);
                KVC_PTR(5, p_seq - 1);
                return true;
            };
            for (uint32_t item_seq = 0; ok;) {
                const int i = take_item(item_seq, false);
                if (i < 0 || i >= a.n_items) break;
                const Item it = decode_item(a, i);
                if (!mbar_wait(&bars[B_QREADY], q_seq & 1, s_abort)) break;
                ++q_seq;
                tc_fence_after();
                if (!issue_s()) break;
                // Q is free once the item's last S MMA completes: the next item's Q loads during this one's tail
                if (it.k0 + 1 == it.k1) umma_commit(&bars[B_QEMPTY]);
                // per key tile: S(k+1), then PV(k)
                for (int k = it.k0; ok && k < it.k1; ++k) {
                    if (k + 1 < it.k1) {
                        if (!issue_s()) { ok = false; break; }
                        if (k + 2 == it.k1) umma_commit(&bars[B_QEMPTY]);
                    }
                    // test hook: a bounded wait on a barrier nothing arrives at, in place of the first
                    // P wait; it gives up after stall_ns (raising the abort flag) with S MMAs in flight
                    if (a.stall_ns != 0 && p_seq == 0) {
                        mbar_wait(&bars[B_STALL], 0, s_abort, a.stall_ns);
                        ok = false;
                        break;
                    }
                    // an item's first PV starts a new O: the softmax has read the previous one out of TMEM
                    // before it signals that P is ready
                    if (!mbar_wait(&bars[B_PFULL], p_seq & 1, s_abort)) { ok = false; break; }
                    ++p_seq;
                    tc_fence_after();
                    if (!issue_pv(k > it.k0)) { ok = false; break; }
                }
            }
            if (*s_abort) {
                // after a wait gave up: let the MMAs in flight finish before TMEM is freed
                volatile int never = 0;
                umma_commit(&bars[B_DRAIN]);
                mbar_wait(&bars[B_DRAIN], 0, &never, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------------------ Q operand (fp16, swizzled)
        // bf16 Q (TMA-loaded) is converted in place; f32 Q is read from global memory; f16 needs nothing.
        constexpr int CPR = D / 8;             // 16-byte chunks per row
        constexpr int RPI = 32 / CPR;          // rows per warp and iteration
        const int cc = lane % CPR, r_off = (warp - 2) * RPI + lane / CPR;
        uint32_t q_seq = 0;
        for (uint32_t item_seq = 0;;) {
            const int i = take_item(item_seq, true);
            if (i < 0 || i >= a.n_items) break;
            const Item it = decode_item(a, i);
            if (!mbar_wait(&bars[B_QFULL], q_seq & 1, s_abort)) break;
            ++q_seq;
            if (QDT != KVC_IN_F16) {
                uint8_t *sQ = sm + L::OFF_Q;
#pragma unroll 4
                for (int r = r_off; r < BM; r += 2 * RPI) {
                    uint4 *p = reinterpret_cast<uint4 *>(sQ + op_off(BM, r, cc));
                    if (QDT == KVC_IN_F32) {
                        const int row = it.qt * BM + r;
                        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                        if (row < a.C) {
                            const float *src = a.q_f32 + ((int64_t)row * a.H_q + it.h) * D + cc * 8;
                            x0 = __ldcg(reinterpret_cast<const float4 *>(src));
                            x1 = __ldcg(reinterpret_cast<const float4 *>(src + 4));
                        }
                        *p = make_uint4(pack_half2(x0.x, x0.y), pack_half2(x0.z, x0.w), pack_half2(x1.x, x1.y),
                                        pack_half2(x1.z, x1.w));
                    } else {
                        const uint4 v = *p;
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[e] = pack_half2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
                        *p = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_QREADY]);
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------------ softmax
        setmaxnreg_inc<L::SM_REGS>();
        const int grp = (warp - 4) >> 2;              // key columns [128 grp, 128 grp + 128) of each tile
        const int r = (warp & 3) * 32 + lane;         // row in the unit = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + COL_S + 128 * grp + lane_base;
        const uint32_t tP = tmem + COL_P + 64 * grp + lane_base;
        const uint32_t tO = tmem + COL_O + (D / 2) * grp + lane_base;
        uint32_t s_seq = 0, o_seq = 0, mb_n = 0;
        bool ok = true;
        const float sl2 = a.scale_log2;
        // The two threads that own a row exchange one float through a mailbox word per (slot, group,
        // row) in shared memory: the value with its lowest mantissa bit replaced by a flag, written and
        // read as one 32-bit word (so no fence is needed).  Exchange n uses slot n & 1 with flag
        // (n >> 1) & 1; a slot is written again only after the partner's next value has been read, which
        // the partner wrote after reading this one, so no value is overwritten unread.  Both threads use
        // the two encoded values (within one ulp of the true ones), so they agree exactly; -inf travels
        // as -FLT_MAX, which every use treats alike.  The wait is bounded.
        auto exchange = [&](float &mine, float &theirs) -> bool {
            const int slot = mb_n & 1;
            const uint32_t flag = (mb_n >> 1) & 1u;
            const int me = (slot * 2 + grp) * BM + r, other = (slot * 2 + (grp ^ 1)) * BM + r;
            mine = fmaxf(mine, -3.402823466e38f);
            const uint32_t enc = (__float_as_uint(mine) & ~1u) | flag;
            mine = __uint_as_float(enc & ~1u);
            s_mb[me] = enc;
            uint32_t w = s_mb[other];
            for (uint32_t n = 0; (w & 1u) != flag; ++n) {
                if ((n & 1023u) == 1023u && (*s_abort || n > (1u << 26))) {
                    *s_abort = 1;
                    return false;
                }
                w = s_mb[other];
            }
            theirs = __uint_as_float(w & ~1u);
            ++mb_n;
            return true;
        };
        for (uint32_t item_seq = 0; ok;) {
            const int i = take_item(item_seq, true);
            if (i < 0 || i >= a.n_items) break;
            const Item it = decode_item(a, i);
            const int row = it.qt * BM + r;       // row within the chunk
            const int t = it.tf + r;              // absolute position
            float m_ref = -INFINITY, l = 0.f;
            for (int k = it.k0; k < it.k1; ++k) {
                if (!mbar_wait(&bars[B_SFULL], s_seq & 1, s_abort)) { ok = false; break; }
                if (threadIdx.x == 128) KVC_PTR(6, s_seq);
                if (threadIdx.x == 256) KVC_PTR(10, s_seq);
                ++s_seq;
                tc_fence_after();
                // my half of the S row in registers (one TMEM round trip), then S may be overwritten
                uint32_t s[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32p(tS + c * 32, s + c * 32);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&bars[B_SFREE]);
                if (threadIdx.x == 128) KVC_PTR(7, s_seq - 1);
                const int key0 = k * BN + 128 * grp;
                if (key0 + 127 > it.tf) {
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (key0 + e > t) s[e] = 0xFF800000u;  // -inf: a key after the query
                }
                // row max: my half in 8 chains of three-input maxima, then the other group's half-row max
                // from the mailbox; both groups take fmaxf(own, other) of the same two values
                float mx8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx8[u] = __uint_as_float(s[u]);
#pragma unroll
                for (int e = 8; e < 120; e += 16) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        mx8[u] = fmax3(mx8[u], __uint_as_float(s[e + u]), __uint_as_float(s[e + 8 + u]));
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(mx8[u], __uint_as_float(s[120 + u]));
                float mx_own =
                    fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                float mx_other;
                if (!exchange(mx_own, mx_other)) { ok = false; break; }
                if (threadIdx.x == 128) KVC_PTR(8, s_seq - 1);
                const float mx = grp == 0 ? fmaxf(mx_own, mx_other) : fmaxf(mx_other, mx_own);
                const float m_new = fmaxf(m_ref, mx * sl2);
                float m_use = m_ref, alpha = 1.f;
                if (k == it.k0) {
                    m_use = m_new;
                } else if (m_new > m_ref + RESCALE_LOG2) {
                    m_use = m_new;
                    alpha = ex2(m_ref - m_new);
                }
                // -inf scores give p = 0 exactly; a row with no visible key so far uses 0 as its offset
                const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;
                // probabilities as fp16 pairs, in three passes over the row so that each pass is a long run
                // of independent operations: exponents by packed fma (in place), 2^x on the MUFU unit (in
                // place), then the row sum (4 packed partial sums, added in a fixed order) and fp16 packing
                const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_sub, -m_sub);
#pragma unroll
                for (int e = 0; e < 128; e += 2) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sl2x2, nm2), x0, x1);
                    s[e] = __float_as_uint(x0);
                    s[e + 1] = __float_as_uint(x1);
                }
#pragma unroll
                for (int e = 0; e < 128; ++e) s[e] = __float_as_uint(ex2(__uint_as_float(s[e])));
                uint32_t pk[64];
                uint64_t rs4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int e = 0; e < 128; e += 2) {
                    const float p0 = __uint_as_float(s[e]), p1 = __uint_as_float(s[e + 1]);
                    rs4[(e >> 1) & 3] = f2_add(rs4[(e >> 1) & 3], f2_pack(p0, p1));
                    pk[e >> 1] = pack_half2(p0, p1);
                }
                float r8[8];
#pragma unroll
                for (int u = 0; u < 4; ++u) f2_unpack(rs4[u], r8[2 * u], r8[2 * u + 1]);
                const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
                l = l * alpha + rs;
                if (k > it.k0) {
                    // P and O are free once PV(k-1) is complete
                    if (!mbar_wait(&bars[B_ODONE], o_seq & 1, s_abort)) { ok = false; break; }
                    ++o_seq;
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                        for (int c = 0; c < D / 64; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + c * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + c * 32, o);
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_st16(tP + c * 16, pk + c * 16);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars[B_PFULL]);
                if (threadIdx.x == 128) KVC_PTR(9, s_seq - 1);
                if (threadIdx.x == 256) KVC_PTR(11, s_seq - 1);
                m_ref = m_use;
            }
            if (!ok) break;
            // ---- epilogue: the row sum over both halves, then O / l or the partial (O, m, l).  The
            // next item's first PV overwrites O only after this thread's next P is published, which
            // comes after these TMEM reads.  A warp stores 32 rows per instruction, so each thread
            // writes 32 bytes at a time (whole sectors) where the buffers are 32-byte aligned.
            if (!mbar_wait(&bars[B_ODONE], o_seq & 1, s_abort)) { ok = false; break; }
            ++o_seq;
            tc_fence_after();
            float l_other;
            if (!exchange(l, l_other)) { ok = false; break; }
            const float l_row = grp == 0 ? l + l_other : l_other + l;
            uint32_t o[D / 2];
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tmem_ld32p(tO + c * 32, o + c * 32);
            tmem_ld_wait();
            if (row < a.C) {
                const int unit = it.qt * a.H_q + it.h;
                float *dst = it.ns == 1 ? a.out + ((int64_t)row * a.H_q + it.h) * D
                                        : a.part + (((int64_t)unit * a.smax + it.s) * BM + r) * PART_ROW(D);
                const float sc = it.ns == 1 ? 1.f / l_row : 1.f;
                float *half = dst + (D / 2) * grp;
                if (a.v8) {
#pragma unroll
                    for (int e = 0; e < D / 2; e += 8)
                        st_global_v8(half + e, __uint_as_float(o[e]) * sc, __uint_as_float(o[e + 1]) * sc,
                                     __uint_as_float(o[e + 2]) * sc, __uint_as_float(o[e + 3]) * sc,
                                     __uint_as_float(o[e + 4]) * sc, __uint_as_float(o[e + 5]) * sc,
                                     __uint_as_float(o[e + 6]) * sc, __uint_as_float(o[e + 7]) * sc);
                } else {
#pragma unroll
                    for (int e = 0; e < D / 2; e += 4)
                        *reinterpret_cast<float4 *>(half + e) =
                            make_float4(__uint_as_float(o[e]) * sc, __uint_as_float(o[e + 1]) * sc,
                                        __uint_as_float(o[e + 2]) * sc, __uint_as_float(o[e + 3]) * sc);
                }
                if (it.ns > 1 && grp == 0) {
                    dst[D] = m_ref;
                    dst[D + 1] = l_row;
                }
            }
        }
    } else if (Q8) {
        // ------------------------------------------------------------------ dequantise
        setmaxnreg_dec<L::DQ_REGS>();
        const int r0 = threadIdx.x - 384;  // key rows r0 and r0 + 128 of each tile
        constexpr int NB = D / 32;
        uint32_t raw_seq = 0, ring_seq = 0;
        bool ok = true;
        auto convert = [&](int kv, int k, int g) -> bool {
            // the scales of my two rows (zero beyond the cache end: TMA zero-fills those codes)
            uint32_t sw[2][NB / 2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int key = k * BN + r0 + 128 * h;
                const uint16_t *sp = (kv ? a.vs : a.ks) + a.layer * a.g.s_layer + (int64_t)key * a.g.s_tok +
                                     g * a.g.s_head;
#pragma unroll
                for (int b = 0; b < NB / 2; ++b) sw[h][b] = 0u;
                if (key < a.kv_len) {
                    if (NB == 4) {
                        const uint2 u = __ldcg(reinterpret_cast<const uint2 *>(sp));
                        sw[h][0] = u.x;
                        sw[h][NB / 2 - 1] = u.y;
                    } else {
                        sw[h][0] = __ldcg(reinterpret_cast<const unsigned int *>(sp));
                    }
                }
            }
            const int st = ring_seq % L::NS;
            if (ring_seq >= (uint32_t)L::NS &&
                !mbar_wait(&bars[B_RING_EMPTY + st], ((ring_seq / L::NS) - 1) & 1, s_abort))
                return false;
            const int rs = raw_seq % L::NR;
            if (!mbar_wait(&bars[B_RAW_FULL + rs], (raw_seq / L::NR) & 1, s_abort)) return false;
            const uint8_t *raw = sm + L::OFF_RAW + rs * L::RAW_BYTES;
            uint8_t *dst = sm + L::OFF_RING + st * L::ST_BYTES;
#pragma unroll 1  // unrolling both rows doubles the code and stalls on instruction fetch
            for (int h = 0; h < 2; ++h) {
                const int rr = r0 + 128 * h;
                uint4 q[D / 16];
#pragma unroll
                for (int c = 0; c < D / 16; ++c)
                    q[c] = *reinterpret_cast<const uint4 *>(raw + ((D == 128) ? sw128(rr, c) : sw64(rr, c)));
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    const int b = c >> 1;
                    const unsigned short sb = (unsigned short)(sw[h][b >> 1] >> (16 * (b & 1)));
                    const __half2 d2 = __halves2half2(__ushort_as_half(sb), __ushort_as_half(sb));
                    uint32_t o[8];
                    dequant4(q[c].x, d2, o[0], o[1]);
                    dequant4(q[c].y, d2, o[2], o[3]);
                    dequant4(q[c].z, d2, o[4], o[5]);
                    dequant4(q[c].w, d2, o[6], o[7]);
                    *reinterpret_cast<uint4 *>(dst + op_off(BN, rr, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(dst + op_off(BN, rr, 2 * c + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
            // order the generic-proxy reads of the raw stage and writes of the operand stage before the
            // async-proxy accesses that follow (the TMA refill, the MMA)
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_RAW_EMPTY + rs]);
            ++raw_seq;
            mbar_arrive(&bars[B_RING_FULL + st]);
            ++ring_seq;
            return true;
        };
        for (uint32_t item_seq = 0; ok;) {
            const int i = take_item(item_seq, true);
            if (i < 0 || i >= a.n_items) break;
            const Item it = decode_item(a, i);
            ok = convert(0, it.k0, it.g);
            for (int k = it.k0; ok && k < it.k1; ++k) {
                if (k + 1 < it.k1) ok = convert(0, k + 1, it.g);
                if (ok) ok = convert(1, k, it.g);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *s_abort) atomicExch(&g_device_status, 1);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Merge of the key splits (merge_row4).  A group of D/4 threads per row, 4 columns each; a block covers
// 256 / (D/4) rows of one unit.
template <int D>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const Args a) {
    // the next kernel (the next chunk's append) may be scheduled now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int TPR = D / 4, RPB = 256 / TPR, BPU = BM / RPB;
    const int rb = blockIdx.x % BPU, unit = blockIdx.x / BPU;
    const int qt = unit / a.H_q, h = unit % a.H_q;
    const int T = unit_tl(a, qt) / BN + 1;
    const int ns = (T + a.ST - 1) / a.ST;
    if (ns <= 1) return;
    // launched as a programmatic dependent of the attention pass: wait until its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int r = rb * RPB + threadIdx.x / TPR, c4 = (threadIdx.x % TPR) * 4;
    const int row = qt * BM + r;
    if (row >= a.C) return;
    const float *base = a.part + ((int64_t)unit * a.smax * BM + r) * PART_ROW(D);
    *reinterpret_cast<float4 *>(a.out + ((int64_t)row * a.H_q + h) * D + c4) =
        merge_row4<D>(base, (int64_t)BM * PART_ROW(D), ns, c4);
}

// ---- q8_0: the attended keys and values dequantised once per call --------------------------
// fp16(d * q) of positions [0, kv_len) of one layer, K (grid.y 0) then V (1), each as [H][n_ctx][D]:
// the very values the in-kernel dequantiser writes into the operand tiles (same op, same rounding),
// so the attention pass then runs as for an f16 cache and gives the same bits.  A thread converts 8
// values (8 code bytes and their block's scale) into 16 bytes.  Launched normally after the append, so
// the append has completed before it starts: it reads the chunk's keys, and its codes and scales are
// read-only for its lifetime (read-only-path loads).  The attention pass may be scheduled as soon as it
// starts.
template <int D>
__global__ void __launch_bounds__(256) dequant_range_kernel(const int8_t *__restrict__ kq,
                                                            const uint16_t *__restrict__ ks,
                                                            const int8_t *__restrict__ vq,
                                                            const uint16_t *__restrict__ vs, Geom g, int layer,
                                                            int kv_len, int n_ctx, int64_t n_units, __half *dk,
                                                            __half *dv) {
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= n_units) return;
    constexpr int UPR = D / 8;                       // 8-value units per head row
    const bool is_v = blockIdx.y != 0;
    const int64_t row = u / UPR;                     // (head, position)
    const int c = (int)(u - row * UPR);
    const int h = (int)(row / kv_len);
    const int t = (int)(row - (int64_t)h * kv_len);
    const int64_t src = layer * g.c_layer + (int64_t)t * g.c_tok + h * g.c_head + 8 * c;
    const uint2 w = __ldg(reinterpret_cast<const uint2 *>((is_v ? vq : kq) + src));
    const uint16_t sb = __ldg((is_v ? vs : ks) + layer * g.s_layer + (int64_t)t * g.s_tok + h * g.s_head + c / 4);
    const __half2 d2 = __halves2half2(__ushort_as_half(sb), __ushort_as_half(sb));
    uint32_t o[4];
    dequant4(w.x, d2, o[0], o[1]);
    dequant4(w.y, d2, o[2], o[3]);
    *reinterpret_cast<uint4 *>((is_v ? dv : dk) + ((int64_t)h * n_ctx + t) * D + 8 * c) =
        make_uint4(o[0], o[1], o[2], o[3]);
}

// ---- the fused step's first kernel --------------------------------------------------------
struct FrontArgs {
    const void *k, *v;     // the chunk's rows, [C][H][D] in the input dtype
    void *kq, *vq;         // the cache's codes (q8_0) or values (f16)
    uint16_t *ks, *vs;     // its scales (q8_0)
    __half *dk, *dv;       // COPY: the fp16 copy, [H][n_ctx][D] each
    Geom g;
    int layer, pos0, H, n_ctx;
    int dq0;               // COPY: the first position converted from the cache (the copy holds [0, dq0))
    int64_t n_dq, n_app;
    unsigned *item_counter;  // the attention pass's item counter, set to zero here
};

// Stores the chunk's K and V at positions [pos0, pos0 + C) exactly as the append kernel does (q8_0
// blocks by the shared quantiser, f16 values rounded to nearest even).  With COPY (q8_0 with the full
// scratch) it also completes the fp16 copy of positions [0, pos0 + C) that the attention pass reads: the
// chunk's from the codes it has just made, positions [dq0, pos0) dequantised from the cache as
// dequant_range_kernel does (the same values either way); [0, dq0) are already there.
// grid.y: K (0) or V (1).  Along x: first n_dq units of 8 earlier values (COPY only), then n_app units
// of the chunk (a 32-value block for q8_0, 8 values for f16).  A programmatic dependent launch: nothing
// global is read or written before griddepcontrol.wait (the previous call's attention pass may still be
// reading the copy).
template <int D, bool Q8, int DT, bool COPY>
__global__ void __launch_bounds__(256) prefill_front_kernel(const FrontArgs f) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the previous call's attention pass has completed (its merge pass waited for it): no CTA still takes
    // items from the counter
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *f.item_counter = 0u;
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool is_v = blockIdx.y != 0;
    const Geom &g = f.g;
    if (COPY && u < f.n_dq) {
        constexpr int UPR = D / 8;                   // 8-value units per head row
        const int64_t row = u / UPR;                 // (head, position) over [dq0, pos0)
        const int c = (int)(u - row * UPR);
        const int nrow = f.pos0 - f.dq0;             // > 0 here: n_dq is zero otherwise
        const int h = (int)(row / nrow), t = f.dq0 + (int)(row - (int64_t)h * nrow);
        const int64_t src = f.layer * g.c_layer + (int64_t)t * g.c_tok + h * g.c_head + 8 * c;
        const uint2 w = __ldcg(reinterpret_cast<const uint2 *>(static_cast<const int8_t *>(is_v ? f.vq : f.kq) + src));
        const uint16_t sb = __ldcg((is_v ? f.vs : f.ks) + f.layer * g.s_layer + (int64_t)t * g.s_tok + h * g.s_head + c / 4);
        const __half2 d2 = __halves2half2(__ushort_as_half(sb), __ushort_as_half(sb));
        uint32_t o[4];
        dequant4(w.x, d2, o[0], o[1]);
        dequant4(w.y, d2, o[2], o[3]);
        *reinterpret_cast<uint4 *>((is_v ? f.dv : f.dk) + ((int64_t)h * f.n_ctx + t) * D + 8 * c) =
            make_uint4(o[0], o[1], o[2], o[3]);
        return;
    }
    const int64_t ua = u - (COPY ? f.n_dq : 0);
    if (ua < 0 || ua >= f.n_app) return;
    const void *in = is_v ? f.v : f.k;
    if constexpr (Q8) {
        constexpr int NB = D / 32;
        const int64_t row = ua / NB;                 // (token, head) in input order
        const int b = (int)(ua - row * NB);
        const int t = (int)(row / f.H), h = (int)(row - (int64_t)t * f.H);
        float x[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float x8[8];
            load_inputs8<DT>(in, row * D + b * 32 + 8 * i, x8);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[8 * i + e] = x8[e];
        }
        uint32_t packed[8];
        const uint16_t scale = q8_0_quantize32(x, packed);
        const int64_t pos = (int64_t)f.pos0 + t;
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<int8_t *>(is_v ? f.vq : f.kq) + f.layer * g.c_layer +
                                               pos * g.c_tok + h * g.c_head + b * 32);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        (is_v ? f.vs : f.ks)[f.layer * g.s_layer + pos * g.s_tok + h * g.s_head + b] = scale;
        if constexpr (COPY) {
            const __half2 d2 = __halves2half2(__ushort_as_half(scale), __ushort_as_half(scale));
            uint32_t o[16];
#pragma unroll
            for (int w = 0; w < 8; ++w) dequant4(packed[w], d2, o[2 * w], o[2 * w + 1]);
            uint4 *cp = reinterpret_cast<uint4 *>((is_v ? f.dv : f.dk) + ((int64_t)h * f.n_ctx + pos) * D + b * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) cp[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
    } else {
        constexpr int UPR = D / 8;
        const int64_t row = ua / UPR;                // (token, head) in input order
        const int c = (int)(ua - row * UPR);
        const int t = (int)(row / f.H), h = (int)(row - (int64_t)t * f.H);
        float x[8];
        load_inputs8<DT>(in, row * D + 8 * c, x);
        const int64_t pos = (int64_t)f.pos0 + t;
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(is_v ? f.vq : f.kq) + f.layer * g.c_layer + pos * g.c_tok +
                                   h * g.c_head + 8 * c) =
            make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]), pack_half2(x[6], x[7]));
    }
}

// ---- host side ----------------------------------------------------------------------
// The work decomposition of one call (see the file comment).
struct Plan {
    int G, n_qt, ST, smax, n_items;
    int cum[MAX_SPLITS + 1], qtmin[MAX_SPLITS];
    size_t part_bytes;   // the key splits' partials
};

// Tiles per split: about a fifth of the cache in steps of 2048 keys, at least 4096 keys, and at
// most MAX_SPLITS splits.  It depends on the cache only, never on the chunk, so a row meets the same
// split boundaries however the prompt is cut.  Shorter splits balance the persistent CTAs better but
// write more partials for the merge (measured: halving the split count from a tenth of the cache
// gained 6% on the late 512-row chunks of a 17k-token f16 prompt and changed nothing on q8_0).
int split_tiles(int n_ctx) {
    int tiles = (n_ctx / 10 + 512) / 1024 * (2048 / BN);
    if (tiles < 4096 / BN) tiles = 4096 / BN;
    const int min_tiles = (n_ctx + MAX_SPLITS * BN - 1) / (MAX_SPLITS * BN);
    return tiles > min_tiles ? tiles : min_tiles;
}

bool make_plan(const kvc_desc &d, int n_head_q, int pos0, int C, Plan &p) {
    p.G = n_head_q / d.n_head_kv;
    p.n_qt = (C + BM - 1) / BM;
    p.ST = split_tiles(d.n_ctx);
    auto T = [&](int qt) {
        const int tl = pos0 + ((qt * BM + BM < C) ? qt * BM + BM : C) - 1;
        return tl / BN + 1;
    };
    p.smax = (T(p.n_qt - 1) + p.ST - 1) / p.ST;
    if (p.smax > MAX_SPLITS) return false;
    p.cum[0] = 0;
    int qt = 0;
    for (int s = 0; s < p.smax; ++s) {
        while (qt < p.n_qt && T(qt) <= s * p.ST) ++qt;
        p.qtmin[s] = qt;
        p.cum[s + 1] = p.cum[s] + (p.n_qt - qt) * n_head_q;
    }
    p.n_items = p.cum[p.smax];
    p.part_bytes = (p.smax > 1) ? (size_t)p.n_qt * n_head_q * p.smax * BM * PART_ROW(d.head_dim) * sizeof(float) : 0;
    return true;
}

// The partials' part of the scratch: a 256-byte header (word 0: prefill_step's item counter), then the
// partials.
constexpr size_t PART_HDR = 256;
size_t scratch_need(const Plan &p) { return PART_HDR + p.part_bytes; }

// scratch: the partials' part of the scratch (header, then partials); counter: null for the static item
// order, else the header's item counter, zeroed by the kernel before this one on the stream.
template <int D, bool Q8, int QDT>
int launch_t(const kvc_cache &c, int layer, int pos0, int n, const void *q, int n_head_q, float *out,
             void *scratch, const Plan &p, cudaStream_t s, unsigned *counter) {
    using L = Cfg<D, Q8>;
    const Geom g = geom_of(c.d);
    const int H = c.d.n_head_kv, kv_len = pos0 + n;
    CUtensorMap tq, tk, tv;
    const uint8_t *kb = static_cast<const uint8_t *>(c.k_q), *vb = static_cast<const uint8_t *>(c.v_q);
    bool ok;
    if (Q8) {
        const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        ok = make_map_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, kb + layer * g.c_layer, D, kv_len, H, g.c_tok,
                         g.c_head, D, BN, 1, sw) &&
             make_map_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, vb + layer * g.c_layer, D, kv_len, H, g.c_tok,
                         g.c_head, D, BN, 1, sw);
    } else {
        ok = make_map_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kb + 2 * layer * g.c_layer, D, kv_len, H,
                         2 * g.c_tok, 2 * g.c_head, 64, BN, 1, CU_TENSOR_MAP_SWIZZLE_128B) &&
             make_map_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, vb + 2 * layer * g.c_layer, D, kv_len, H,
                         2 * g.c_tok, 2 * g.c_head, 64, BN, 1, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!ok) return KVC_ECUDA;
    if (QDT != KVC_IN_F32) {
        const CUtensorMapDataType dt =
            QDT == KVC_IN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if (!make_map_3d(&tq, dt, q, D, n_head_q, n, (uint64_t)D * 2, (uint64_t)n_head_q * D * 2, 64, 1, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KVC_ECUDA;
    } else {
        tq = tk;  // unused by the f32 variant
    }
    Args a;
    a.q_f32 = QDT == KVC_IN_F32 ? static_cast<const float *>(q) : nullptr;
    a.ks = static_cast<const uint16_t *>(c.k_s);
    a.vs = static_cast<const uint16_t *>(c.v_s);
    a.out = out;
    a.part = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) + PART_HDR);
    a.item_counter = counter;
    a.v8 = ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(a.part)) & 31) == 0;
    a.g = g;
    a.layer = layer;
    a.pos0 = pos0;
    a.C = n;
    a.kv_len = kv_len;
    a.H_q = n_head_q;
    a.G = p.G;
    a.H_kv = H;
    a.n_qt = p.n_qt;
    a.ST = p.ST;
    a.smax = p.smax;
    a.n_items = p.n_items;
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)D));
    a.stall_ns = take_test_stall(KVC_TEST_PREFILL);
    for (int i = 0; i <= MAX_SPLITS; ++i) a.cum[i] = i <= p.smax ? p.cum[i] : p.n_items;
    for (int i = 0; i < MAX_SPLITS; ++i) a.qtmin[i] = i < p.smax ? p.qtmin[i] : p.n_qt;
    auto kern = prefill_kernel<D, Q8, QDT>;
    if (allow_dynamic_smem((const void *)kern, L::ALLOC) != KVC_OK) return KVC_ECUDA;
    const int grid = p.n_items < sm_count() ? p.n_items : sm_count();
    // both passes may be scheduled while the kernel before them finishes; each waits for it on the
    // device before it touches global memory
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(L::THREADS);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a) != cudaSuccess) return KVC_ECUDA;
    if (p.smax > 1) {
        constexpr int BPU = BM / (256 / (D / 4));
        cudaLaunchConfig_t cfg2 = {};
        cfg2.gridDim = dim3(p.n_qt * n_head_q * BPU);
        cfg2.blockDim = dim3(256);
        cfg2.dynamicSmemBytes = 0;
        cfg2.stream = s;
        cfg2.attrs = attr;
        cfg2.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg2, prefill_merge_kernel<D>, a) != cudaSuccess) return KVC_ECUDA;
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

template <int D, bool Q8>
int launch_d(const kvc_cache &c, int layer, int pos0, int n, const void *q, int dtype, int n_head_q,
             float *out, void *scratch, const Plan &p, cudaStream_t s, unsigned *counter = nullptr) {
    switch (dtype) {
        case KVC_IN_F32:
            return launch_t<D, Q8, KVC_IN_F32>(c, layer, pos0, n, q, n_head_q, out, scratch, p, s, counter);
        case KVC_IN_BF16:
            return launch_t<D, Q8, KVC_IN_BF16>(c, layer, pos0, n, q, n_head_q, out, scratch, p, s, counter);
        default:
            return launch_t<D, Q8, KVC_IN_F16>(c, layer, pos0, n, q, n_head_q, out, scratch, p, s, counter);
    }
}

// The fused step's first kernel for one variant (programmatic dependent launch).
template <int D, bool Q8, int DT, bool COPY>
int launch_front_t(const FrontArgs &f, cudaStream_t s) {
    const int64_t units = (COPY ? f.n_dq : 0) + f.n_app;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((units + 255) / 256), 2);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_front_kernel<D, Q8, DT, COPY>, f) == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

template <int D, bool Q8, bool COPY>
int launch_front_d(const FrontArgs &f, int dtype, cudaStream_t s) {
    switch (dtype) {
        case KVC_IN_F32: return launch_front_t<D, Q8, KVC_IN_F32, COPY>(f, s);
        case KVC_IN_BF16: return launch_front_t<D, Q8, KVC_IN_BF16, COPY>(f, s);
        default: return launch_front_t<D, Q8, KVC_IN_F16, COPY>(f, s);
    }
}

int launch_front(const FrontArgs &f, int D, bool q8, bool copy, int dtype, cudaStream_t s) {
    if (D == 128)
        return !q8 ? launch_front_d<128, false, false>(f, dtype, s)
                   : copy ? launch_front_d<128, true, true>(f, dtype, s) : launch_front_d<128, true, false>(f, dtype, s);
    return !q8 ? launch_front_d<64, false, false>(f, dtype, s)
               : copy ? launch_front_d<64, true, true>(f, dtype, s) : launch_front_d<64, true, false>(f, dtype, s);
}

}  // namespace

// q8_0: bytes of the fp16 copy of one layer's keys and values (capacity n_ctx positions)
size_t dequant_copy_bytes(const kvc_desc &d) {
    return d.type == KVC_Q8_0 ? (size_t)2 * d.n_head_kv * d.n_ctx * d.head_dim * sizeof(__half) : 0;
}

size_t prefill_scratch_bytes(const kvc_desc &d, int n_head_q, int max_tokens) {
    // the largest plan over chunk positions: q-tiles grow with the chunk, splits with the context
    Plan p;
    if (!make_plan(d, n_head_q, d.n_ctx - max_tokens, max_tokens, p)) return 0;
    return dequant_copy_bytes(d) + scratch_need(p);
}


int launch_prefill(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *q, int dtype,
                   int n_head_q, float *out, void *scratch, size_t scratch_bytes, cudaStream_t s) {
    if (n_tokens == 0) return KVC_OK;
    Plan p;
    if (!make_plan(c.d, n_head_q, pos0, n_tokens, p)) return KVC_EINVAL;
    if (scratch_need(p) > scratch_bytes) return KVC_ENOSPC;
    const bool q8 = c.d.type == KVC_Q8_0;
    const size_t copy_bytes = dequant_copy_bytes(c.d);
    if (q8 && scratch_bytes >= copy_bytes + scratch_need(p)) {
        // the attended keys and values dequantised once into the scratch, then attention as for an f16
        // cache laid out [head][position][D]; the plan (key splits) stays the q8_0 cache's own
        const int kv_len = pos0 + n_tokens, H = c.d.n_head_kv, D = c.d.head_dim;
        __half *dk = static_cast<__half *>(scratch);
        __half *dv = dk + (size_t)H * c.d.n_ctx * D;
        const int64_t n_units = (int64_t)H * kv_len * (D / 8);
        const dim3 grid((unsigned)((n_units + 255) / 256), 2);
        const Geom g = geom_of(c.d);
        if (D == 128)
            dequant_range_kernel<128><<<grid, 256, 0, s>>>(static_cast<const int8_t *>(c.k_q),
                                                           static_cast<const uint16_t *>(c.k_s),
                                                           static_cast<const int8_t *>(c.v_q),
                                                           static_cast<const uint16_t *>(c.v_s), g, layer, kv_len,
                                                           c.d.n_ctx, n_units, dk, dv);
        else
            dequant_range_kernel<64><<<grid, 256, 0, s>>>(static_cast<const int8_t *>(c.k_q),
                                                          static_cast<const uint16_t *>(c.k_s),
                                                          static_cast<const int8_t *>(c.v_q),
                                                          static_cast<const uint16_t *>(c.v_s), g, layer, kv_len,
                                                          c.d.n_ctx, n_units, dk, dv);
        kvc_cache f = {};
        f.d = c.d;
        f.d.n_layer = 1;
        f.d.n_ctx = c.d.n_ctx;
        f.d.type = KVC_F16;
        f.d.layout = KVC_HEAD_MAJOR;
        f.k_q = dk;
        f.v_q = dv;
        void *part = static_cast<uint8_t *>(scratch) + copy_bytes;
        return D == 128 ? launch_d<128, false>(f, 0, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s)
                        : launch_d<64, false>(f, 0, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s);
    }
    if (c.d.head_dim == 128)
        return q8 ? launch_d<128, true>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, scratch, p, s)
                  : launch_d<128, false>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, scratch, p, s);
    return q8 ? launch_d<64, true>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, scratch, p, s)
              : launch_d<64, false>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, scratch, p, s);
}

int launch_prefill_step(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *q, const void *k,
                        const void *v, int dtype, int n_head_q, float *out, void *scratch, size_t scratch_bytes,
                        int copy_valid, cudaStream_t s) {
    if (n_tokens == 0) return KVC_OK;
    Plan p;
    if (!make_plan(c.d, n_head_q, pos0, n_tokens, p)) return KVC_EINVAL;
    if (scratch_need(p) > scratch_bytes) return KVC_ENOSPC;
    const bool q8 = c.d.type == KVC_Q8_0;
    const size_t copy_bytes = dequant_copy_bytes(c.d);
    const bool copy = q8 && scratch_bytes >= copy_bytes + scratch_need(p);
    const int H = c.d.n_head_kv, D = c.d.head_dim;
    uint8_t *part = static_cast<uint8_t *>(scratch) + (copy ? copy_bytes : 0);
    FrontArgs f;
    f.k = k;
    f.v = v;
    f.kq = c.k_q;
    f.vq = c.v_q;
    f.ks = static_cast<uint16_t *>(c.k_s);
    f.vs = static_cast<uint16_t *>(c.v_s);
    f.dk = copy ? static_cast<__half *>(scratch) : nullptr;
    f.dv = copy ? f.dk + (size_t)H * c.d.n_ctx * D : nullptr;
    f.g = geom_of(c.d);
    f.layer = layer;
    f.pos0 = pos0;
    f.H = H;
    f.n_ctx = c.d.n_ctx;
    f.dq0 = copy ? copy_valid : 0;
    f.n_dq = copy ? (int64_t)H * (pos0 - f.dq0) * (D / 8) : 0;
    f.n_app = (int64_t)n_tokens * H * (q8 ? D / 32 : D / 8);
    f.item_counter = reinterpret_cast<unsigned *>(part);
    // the chunk stored (and, with the copy, the attended range in fp16), then the attention and the merge
    const int rc = launch_front(f, D, q8, copy, dtype, s);
    if (rc != KVC_OK) return rc;
    // the attention pass takes its items from the counter the front kernel has just zeroed: a CTA that
    // finishes early takes the next item in order, and the order keeps concurrent CTAs on the same tiles
    unsigned *ctr = f.item_counter;
    if (copy) {
        kvc_cache fc = {};
        fc.d = c.d;
        fc.d.n_layer = 1;
        fc.d.n_ctx = c.d.n_ctx;
        fc.d.type = KVC_F16;
        fc.d.layout = KVC_HEAD_MAJOR;
        fc.k_q = f.dk;
        fc.v_q = f.dv;
        return D == 128 ? launch_d<128, false>(fc, 0, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s, ctr)
                        : launch_d<64, false>(fc, 0, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s, ctr);
    }
    if (D == 128)
        return q8 ? launch_d<128, true>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s, ctr)
                  : launch_d<128, false>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s, ctr);
    return q8 ? launch_d<64, true>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s, ctr)
              : launch_d<64, false>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, part, p, s, ctr);
}

int read_and_clear_device_status(int32_t *status) {
    if (cudaDeviceSynchronize() != cudaSuccess) return KVC_ECUDA;
    int v = 0, dv = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return KVC_ECUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return KVC_ECUDA;
    if (read_and_clear_decode_status(&dv) != KVC_OK) return KVC_ECUDA;
    *status = v ? v : dv;
    return KVC_OK;
}

}  // namespace kvc

#ifdef KVC_TRACE
// Diagnostic build only: clear, or copy out (16 x 128 uint64), the attention pass's clock stamps.
extern "C" int kvc_ptrace_clear() {
    static unsigned long long z[16 * 128] = {};
    return cudaMemcpyToSymbol(kvc::g_ptrace, z, sizeof(z)) == cudaSuccess ? 0 : -1;
}
extern "C" int kvc_ptrace_read(unsigned long long *host) {
    return cudaMemcpyFromSymbol(host, kvc::g_ptrace, sizeof(kvc::g_ptrace)) == cudaSuccess ? 0 : -1;
}
#endif
