// attn_verify_tc.cu -- attention tree verify on the 5th-generation tensor
// cores (tcgen05 + tensor memory), head sizes 128 and 256.
//
// What it computes is the attention step of include/dflv.h ("Luce DFlash"
// README, "How it works": one target pass verifies the tree through a causal
// mask derived from parent pointers; "--fa-window N"; "Asymmetric K/V
// quantization": q8_0 default, Q4_0): the tree's keys/values are quantised
// into cache slots [P, P + n), and every (node, query head) attends to the
// cached positions inside its window and to its ancestors-or-self.
//
// How: one thread-block cluster per (sequence, KV head, row tile of <= 128
// query rows); the cluster's CTAs split the visible cache keys into 32-key
// tiles (tile starts aligned to 32 keys) by cost, and the tree block is one
// or two extra tiles.  Inside a CTA the tiles flow through a pipeline of
// warp roles that hand over through mbarriers (every wait bounded):
//   * load warps (2, one per plane): the raw codes and scales of each tile
//     by bulk copies (TMA engine) into double buffers, completion counted in
//     bytes on an mbarrier; the first two tiles are requested before the kernel waits
//     for its predecessor when early prefetch is on (and, when every cluster
//     of the launch is resident at once, L2 requests for the layer's query
//     rows and the tree's new keys and values).  The CTA that attends to a
//     tree tile first quantises the tree's rows into the cache;
//   * stage warps (4): each raw tile is expanded into fp16 hi + lo tiles
//     with the block scale folded in (d * code is exact in fp32; hi =
//     fp16(x), lo = fp16(x - hi)).  K and V tiles are double-buffered;
//   * the MMA warp (1) issues tcgen05.mma: [S_hi | S_lo] = Q [K_hi ; K_lo]^T
//     into the S buffer in tensor memory (M = 128, N = 64, K = head size),
//     and O += P_hi V_hi + P_hi V_lo + P_lo V_hi with O resident in tensor
//     memory.  Q and P are read from tensor memory, so the tensor core's
//     shared-memory reads are only the K and V tiles.  Per tile t it issues
//     tile t+1's scores as soon as the softmax has read tile t's, then tile
//     t's products once P is written (two P buffers);
//   * softmax warps (4): one thread per query row (its TMEM lane) writes the
//     row's query into tensor memory once, then per tile reads the 32
//     scores, applies the tree / window mask and an fp32 online softmax with
//     a lazily updated running max (O is rescaled in tensor memory only when
//     a row's max grows by more than 2^8), and writes P as fp16 hi + lo.
// Partial (max, sum, O) are merged across the cluster: with a caller's
// workspace through global memory (each CTA writes its rows' partials, one
// cluster barrier, then every CTA merges an even share of the outputs), else
// through distributed shared memory.  Operands use the no-swizzle
// core-matrix layout described in tcgen05.cuh.
#include <climits>

#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "tree.cuh"

namespace dflv {

namespace {

using namespace attn;

constexpr int kTK = 32;          // keys per tile
constexpr int kRows = 128;       // MMA M: query rows per CTA
constexpr int kSoftWarps = 4;    // warps 0-3
constexpr int kStageWarps = 4;   // warps 4-7
constexpr int kMmaWarp = kSoftWarps + kStageWarps;  // warp 8
constexpr int kLoadWarp = kMmaWarp + 1;              // warp 9: raw K tile copies, warp 10: raw V
constexpr int kThreads = (kLoadWarp + 2) * 32;
constexpr int kStage0 = kSoftWarps * 32;             // first stage thread
constexpr int kStageThreads = kStageWarps * 32;
constexpr int kStageBarrier = 2;                     // named barrier of the stage warps
constexpr int kPrepBarrier = 3;                      // named barrier of the other warps (Q, tree rows)
constexpr int kPrepThreads = kThreads - kStageThreads;
constexpr int kTreeCost = 3;                         // a tree tile (quantise + attend) in cache tiles

// One raw plane (codes + scales of kTK keys) in the format T.
template <int D, int T>
struct PlaneFmt {
    static constexpr int NB = D / 32;
    static constexpr int KB = (T == DFLV_KV_Q8_0) ? D : (T == DFLV_KV_TQ3_0) ? D / 32 * 12 : D / 2;  // code bytes per key row
    static constexpr int RSK = KB + 16;                            // padded raw row stride
    static constexpr size_t kRawCodes = (size_t)kTK * RSK;
    static constexpr size_t kRawScales = (size_t)kTK * NB * 2 + 16;  // + room for a misaligned start
    static constexpr size_t kRaw = kRawCodes + kRawScales;           // one plane of one tile
    static_assert(kRawCodes % 16 == 0 && kRaw % 16 == 0, "copy destinations stay 16-byte aligned");
};

// Keys in format KT, values in format VT (equal unless the cache is
// asymmetric).
template <int D, int KT, int VT>
struct TcLayout {
    using FK = PlaneFmt<D, KT>;
    using FV = PlaneFmt<D, VT>;
    static constexpr int NB = D / 32;
    static constexpr int OS = D + 4;                                  // merge row stride (floats)
    static constexpr size_t kHeader = 2048;   // tree arrays, barriers, flags
    static constexpr size_t kK = (size_t)2 * kTK * D * 2;    // K_hi rows 0-31, K_lo rows 32-63
    static constexpr size_t kV = (size_t)kTK * D * 2;        // one of V_hi, V_lo
    static constexpr size_t off_K = kHeader;                 // two buffers
    static constexpr size_t off_V = off_K + 2 * kK;          // two buffers of V_hi then V_lo
    static constexpr size_t off_rawK = off_V + 4 * kV;           // two buffers
    static constexpr size_t off_rawV = off_rawK + 2 * FK::kRaw;  // two buffers
    // TQ3_0: the rotated query rows of one half of the row tile, fp16
    static constexpr bool kRotated = KT == DFLV_KV_TQ3_0;
    static constexpr size_t off_QS = off_rawV + 2 * FV::kRaw;
    static constexpr size_t kQS = kRotated ? (size_t)(kRows / 2) * (D + 8) * 2 : 0;  // row stride D + 8 halves
    static constexpr size_t loop_total = off_QS + kQS;
    // merge: CS x ceil(RT / CS) <= kRows + 15 received partial rows
    static constexpr size_t off_Om = kHeader;
    static constexpr size_t merge_total = off_Om + (size_t)(kRows + 16) * OS * 4;
    static constexpr size_t total = loop_total > merge_total ? loop_total : merge_total;
    // tensor memory: O in columns [0, D), the S buffer ([S_hi | S_lo], 2 kTK
    // columns) at kScol, two P buffers of kTK columns (P_hi | P_lo as fp16
    // pairs) at kPcol, Q (fp16 pairs) in D / 2 columns at kQcol
    static constexpr uint32_t kScol = D, kPcol = D + 2 * kTK, kQcol = D + 4 * kTK;
    static constexpr uint32_t kTmemCols = (kQcol + D / 2 <= 256) ? 256 : 512;
    static_assert(kQcol + D / 2 <= 512, "O, the S buffers and Q fit in tensor memory");
};

// header offsets
constexpr int kHdrDepth = 256, kHdrMask = 512, kHdrBar = 1024, kHdrSlot = 1280, kHdrFail = 1284;
enum Bar { kRawK0, kRawK1, kRawV0, kRawV1, kKFree0, kKFree1, kVFree0, kVFree1, kKReady0, kKReady1, kVReady0,
           kVReady1, kSFull0, kSFull1, kSFree0, kSFree1, kPReady0, kPReady1, kODone0, kODone1, kMmaFin, kNumBars };
static_assert(kHdrBar + kNumBars * 8 <= kHdrSlot, "barriers fit below the TMEM slot");

DFLV_DEVINL bool wait_phase(uint64_t* bar, uint32_t parity) {
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---------------------------------------------------------------- TQ3_0
// Eight three-bit codes (bits 3j .. 3j+2 of `bits`) -> value - 4 as exact
// fp16 pairs: 0x6400 | c is 1024 + c.
DFLV_DEVINL void u3x8_to_f16x2(uint32_t bits, uint32_t (&cv)[4]) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6404), __ushort_as_half(0x6404));  // 1028
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t c0 = (bits >> (6 * e)) & 7u, c1 = (bits >> (6 * e + 3)) & 7u;
        const uint32_t w = 0x64006400u | c0 | (c1 << 16);
        const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&w), bias);
        cv[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
}

// Orthonormal Walsh-Hadamard transform (Sylvester order) of one row of D
// values held by a warp, D/32 consecutive values per lane: the butterflies
// (a + b, a - b on the pair (j, j + h)) with strides h = 1, 2, ..., D/2 in
// that order, then the product with fl(1/sqrt(D)).  These are the fp32
// operations of the plain serial loop, in its order for every element, so
// the result is bit-identical to it.
template <int D>
DFLV_DEVINL void fwht_warp(float (&v)[D / 32], int lane) {
    constexpr int V = D / 32;
#pragma unroll
    for (int h = 1; h < V; h *= 2)
#pragma unroll
        for (int j = 0; j < V; ++j)
            if ((j & h) == 0) {
                const float x = v[j], y = v[j + h];
                v[j] = __fadd_rn(x, y);
                v[j + h] = __fsub_rn(x, y);
            }
#pragma unroll
    for (int hl = 1; hl < 32; hl *= 2) {  // stride h = hl * V: the partner lane holds the other element
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const float o = __shfl_xor_sync(0xffffffffu, v[j], hl);
            v[j] = (lane & hl) ? __fsub_rn(o, v[j]) : __fadd_rn(v[j], o);
        }
    }
    const float s = (float)(1.0 / sqrt((double)D));
#pragma unroll
    for (int j = 0; j < V; ++j) v[j] = __fmul_rn(v[j], s);
}

// A bf16 row of D values -> the warp's registers (D/32 consecutive per lane).
template <int D>
DFLV_DEVINL void load_row_warp(const uint16_t* src, float (&v)[D / 32], int lane) {
    constexpr int V = D / 32;
    uint32_t w[V / 2];
    if constexpr (V == 8) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(src) + lane);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else {
        const uint2 x = __ldg(reinterpret_cast<const uint2*>(src) + lane);
        w[0] = x.x; w[1] = x.y;
    }
#pragma unroll
    for (int e = 0; e < V / 2; ++e) {
        v[2 * e] = bf16_bits_to_float((uint16_t)(w[e] & 0xffff));
        v[2 * e + 1] = bf16_bits_to_float((uint16_t)(w[e] >> 16));
    }
}

// One rotated tree row into the TQ3_0 cache: the warp's D values (after
// fwht_warp) in blocks of 32 (32 / V lanes each): d = amax / 3 stored as
// fp16, codes = clamp(round-half-away(x * fl(1/d)), -4, 3) + 4 packed as a
// little-endian bit stream of 3 bits per value, 12 bytes per block.
template <int D>
DFLV_DEVINL void quantize_tq3_warp(const float (&v)[D / 32], uint8_t* __restrict__ codes,
                                   uint16_t* __restrict__ scales, int lane) {
    constexpr int V = D / 32, LPB = 32 / V;  // values per lane, lanes per block
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < V; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
    for (int o = 1; o < LPB; o *= 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 3.f);
    const float id = (d != 0.f) ? __frcp_rn(d) : 0.f;
    uint32_t bits = 0;
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int c = (int)fminf(fmaxf(roundf(__fmul_rn(v[j], id)), -4.f), 3.f) + 4;
        bits |= (uint32_t)c << (3 * j);
    }
    const int blk = lane / LPB, q = lane % LPB;
    if constexpr (V == 4) {
        // 12 bits per lane: even lanes take their odd neighbour's bits and
        // write the pair's 3 bytes
        const uint32_t nb = __shfl_down_sync(0xffffffffu, bits, 1);
        if ((q & 1) == 0) {
            bits |= nb << 12;
            uint8_t* p = codes + blk * 12 + 3 * (q / 2);
            p[0] = (uint8_t)bits;
            p[1] = (uint8_t)(bits >> 8);
            p[2] = (uint8_t)(bits >> 16);
        }
    } else {
        uint8_t* p = codes + blk * 12 + 3 * q;
        p[0] = (uint8_t)bits;
        p[1] = (uint8_t)(bits >> 8);
        p[2] = (uint8_t)(bits >> 16);
    }
    if (q == 0) scales[blk] = __half_as_ushort(__float2half_rn(d));
}

// Expand one raw tile (codes + scales of `count` keys) into fp16 hi + lo with
// the block scale d folded in; rows past count are zero.  Codes become exact
// fp16 values by byte permutation; hi = d * code rounded once (HMUL2) and
// lo = d * code - hi rounded once (HFMA2: the fused product is exact), the
// same bits as rounding the exact fp32 product and its remainder.  The 128
// stage threads take items key % 8 fastest, so 8 consecutive threads fill
// one 128-byte core-matrix run.
template <int D, int TYPE>
DFLV_DEVINL void stage_hilo(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int count,
                            uint8_t* __restrict__ hi, uint8_t* __restrict__ lo, int st) {
    using L = PlaneFmt<D, TYPE>;
    constexpr int C8 = D / 8;
    constexpr int PER = kTK * C8 / kStageThreads;  // items per thread
    static_assert(PER * kStageThreads == kTK * C8, "items split evenly over the stage threads");
    uint2 wv[PER];
    uint16_t sbv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {  // every load first
        const int idx = st + j * kStageThreads;
        const int c = (idx & 7) + (idx / (8 * C8)) * 8, d8 = (idx >> 3) % C8;
        wv[j] = make_uint2(0, 0);
        sbv[j] = 0;
        if (c < count) {
            sbv[j] = scales[c * L::NB + (d8 * 8) / 32];
            if constexpr (TYPE == DFLV_KV_Q8_0) {
                wv[j] = *reinterpret_cast<const uint2*>(codes + c * L::RSK + d8 * 8);
            } else if constexpr (TYPE == DFLV_KV_TQ3_0) {
                // the 8 three-bit codes of this chunk: 3 whole bytes
                const uint8_t* p = codes + c * L::RSK + (d8 / 4) * 12 + 3 * (d8 % 4);
                wv[j].x = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16);
            } else {
                const int blk = (d8 * 8) / 32, off = (d8 * 8) % 32;
                wv[j] = *reinterpret_cast<const uint2*>(codes + c * L::RSK + blk * 16 + (off & 15));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int idx = st + j * kStageThreads;
        const int c = (idx & 7) + (idx / (8 * C8)) * 8;  // key
        const int d8 = (idx >> 3) % C8;                    // 8-dim chunk
        uint4 h = make_uint4(0, 0, 0, 0), l = make_uint4(0, 0, 0, 0);
        if (c < count) {
            const __half2 d2 = __halves2half2(__ushort_as_half(sbv[j]), __ushort_as_half(sbv[j]));
            uint32_t cv[4];  // 8 codes as 4 half2
            const uint2 w = wv[j];
            if constexpr (TYPE == DFLV_KV_Q8_0) {
                i8x4_to_f16x2(w.x, cv[0], cv[1]);
                i8x4_to_f16x2(w.y, cv[2], cv[3]);
            } else if constexpr (TYPE == DFLV_KV_TQ3_0) {
                u3x8_to_f16x2(w.x, cv);
            } else {
                // element j < 16 of a 32-block in the low nibble of byte j,
                // element j + 16 in its high nibble
                const int off = (d8 * 8) % 32;
                const uint32_t m0 = off >= 16 ? (w.x >> 4) & 0x0f0f0f0fu : w.x & 0x0f0f0f0fu;
                const uint32_t m1 = off >= 16 ? (w.y >> 4) & 0x0f0f0f0fu : w.y & 0x0f0f0f0fu;
                u4x4_to_f16x2(m0, cv[0], cv[1]);
                u4x4_to_f16x2(m1, cv[2], cv[3]);
            }
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __half2 x = *reinterpret_cast<const __half2*>(&cv[e]);
                const __half2 h2 = __hmul2(x, d2);
                const __half2 l2 = __hfma2(x, d2, __hneg2(h2));
                hv[e] = *reinterpret_cast<const uint32_t*>(&h2);
                lv[e] = *reinterpret_cast<const uint32_t*>(&l2);
            }
            h = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            l = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
        const uint32_t off = tc::cm_offset(c, d8 * 8, D);
        *reinterpret_cast<uint4*>(hi + off) = h;
        *reinterpret_cast<uint4*>(lo + off) = l;
    }
}

// One raw plane (codes + scales) of a cache tile is requested by the 32 lanes
// of a load warp with bulk copies (see issue_raw); bar is initialised for
// 32 arrivals and the copied bytes.  The scales are copied from the 16-byte
// boundary at or below the first one (their byte offset in the buffer is
// returned by scale_shift).
template <int D, int TYPE>
DFLV_DEVINL int scale_shift(const uint16_t* plane_scales, size_t row0, int start) {
    using L = PlaneFmt<D, TYPE>;
    return (int)(reinterpret_cast<uintptr_t>(plane_scales + (row0 + start) * L::NB) & 15);
}

template <int D, int TYPE>
DFLV_DEVINL void issue_raw(const uint8_t* plane_codes, const uint16_t* plane_scales, size_t row0, int start,
                           int count, uint8_t* raw, uint64_t* bar, int st) {
    using L = PlaneFmt<D, TYPE>;
    // bulk copies (TMA engine): one per key row (into the padded row
    // stride) by the warp's lanes, one for the scales; the barrier expects
    // the warp's 32 arrivals and the bytes
    const uintptr_t sa = reinterpret_cast<uintptr_t>(plane_scales + (row0 + start) * L::NB);
    const int shift = (int)(sa & 15);
    const uint32_t sbytes = (uint32_t)((shift + count * L::NB * 2 + 15) >> 4) * 16;
    if (st == 0) mbar_arrive_expect_tx(bar, (uint32_t)(count * L::KB) + sbytes);
    else mbar_arrive(bar);
    for (int c = st; c < count; c += 32)
        bulk_g2s(raw + c * L::RSK, plane_codes + (row0 + start + c) * L::KB, L::KB, bar);
    if (st == 0) bulk_g2s(raw + L::kRawCodes, reinterpret_cast<const void*>(sa - shift), sbytes, bar);
}

// barrier over `count` threads (whole warps) under id
DFLV_DEVINL void named_barrier_sync_n(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// barrier over `count` threads (whole warps) under id; returns the OR of
// pred over them, the same value in every participating thread
DFLV_DEVINL bool named_barrier_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

struct TileInfo {
    int start, count;
    bool tree;
};

template <int D, int KT, int VT>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnVerifyArgs a, int RT, int CS) {
    using L = TcLayout<D, KT, VT>;
    using FK = typename L::FK;
    using FV = typename L::FV;
    constexpr int NB = L::NB, OS = L::OS;
    extern __shared__ __align__(1024) unsigned char smem[];
    int32_t* par_s = reinterpret_cast<int32_t*>(smem);
    int32_t* depth_s = reinterpret_cast<int32_t*>(smem + kHdrDepth);
    uint64_t* amask_s = reinterpret_cast<uint64_t*>(smem + kHdrMask);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kHdrBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kHdrSlot);
    int32_t* fail_s = reinterpret_cast<int32_t*>(smem + kHdrFail);
    auto failed = [&]() { return *reinterpret_cast<volatile int32_t*>(fail_s) != 0; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int kvh = blockIdx.y % a.Hkv, rt = blockIdx.y / a.Hkv, b = blockIdx.z;
    const int G = a.Hq / a.Hkv, N = a.N_max, W = a.window;
    const bool early = (a.flags & DFLV_FLAG_EARLY_PREFETCH) != 0;

    // Before the dependency wait (early prefetch) only the tree, n_past and
    // the cached slots below P are read; none of them is written by the
    // kernel this one may overlap.
    if (!early) grid_dependency_wait();
    const int n = __ldg(a.n_nodes + b), P = __ldg(a.n_past + b);
    // Uniform over the cluster: every CTA leaves before any cluster barrier.
    if (P < 0 || P + n > a.cap || n < 1 || n > N) {
        if (tid == 0 && rank == 0 && rt == 0 && kvh == 0)
            raise_status(a.status, (n < 1 || n > N) ? DFLV_DEV_TOPOLOGY : DFLV_DEV_CAPACITY);
        return;
    }
    const int rows_valid = G * n, row0 = rt * RT;
    if (row0 >= rows_valid) return;
    if (!block_tree_topology(a.parent + (size_t)b * N, n, N, par_s, depth_s, amask_s,
                             (rank == 0 && rt == 0 && kvh == 0) ? a.status : nullptr))
        return;  // uniform over the cluster: the parent array is shared

    const size_t plane_row0 = ((size_t)b * a.Hkv + kvh) * a.cap;
    uint8_t* kq = reinterpret_cast<uint8_t*>(a.kq);
    uint8_t* vq = reinterpret_cast<uint8_t*>(a.vq);

    // tiles: visible cache keys [lo, P) in 32-key tiles starting at a
    // multiple of 32, then the tree slots [P, P + n).  The list is split over
    // the cluster by cost, a tree tile counting kTreeCost cache tiles (its
    // CTA also quantises it), so the tree tiles go to the last ranks
    const int lo = (W > 0) ? max(0, P - W + 1) : 0;
    const int c0 = (lo / kTK) * kTK;
    const int n_cache_tiles = (P > lo) ? (P - c0 + kTK - 1) / kTK : 0;
    const int n_tree_tiles = (n + kTK - 1) / kTK;
    const int n_all = n_cache_tiles + n_tree_tiles;
    const long total_cost = (long)n_cache_tiles + (long)kTreeCost * n_tree_tiles;
    auto tile_at_cost = [&](long c) {  // first tile whose cumulative cost reaches c
        return (int)(c <= n_cache_tiles ? c : n_cache_tiles + (c - n_cache_tiles + kTreeCost - 1) / kTreeCost);
    };
    const int g0 = tile_at_cost(total_cost * rank / CS);
    const int T = min(n_all, tile_at_cost(total_cost * (rank + 1) / CS)) - g0;
    auto tile = [&](int u) {
        const int g = g0 + u;
        TileInfo ti;
        ti.tree = g >= n_cache_tiles;
        ti.start = ti.tree ? P + (g - n_cache_tiles) * kTK : c0 + g * kTK;
        ti.count = ti.tree ? min(kTK, P + n - ti.start) : min(kTK, P - ti.start);
        return ti;
    };
    // With early prefetch in a launch whose clusters are all resident at
    // once, the layer inputs this CTA reads after the dependency wait -- its
    // query rows and, where it quantises tree rows, their new keys and
    // values -- are first asked for in the L2 (in a model the layer before
    // has just written them there); the loads after the wait read whatever
    // the lines hold by then.
    if (a.flags & kFlagPrefetchInputs) {
        const int nq = min(RT, rows_valid - row0);
        const int t_lo = max(0, g0 - n_cache_tiles) * kTK, t_hi = min(n, (g0 + T - n_cache_tiles) * kTK);
        const int nt = t_hi > t_lo ? t_hi - t_lo : 0;
        for (int k = tid; k < nq + 2 * nt; k += (int)blockDim.x) {
            if (k < nq) {
                const int rho = row0 + k;
                prefetch_l2_bulk(a.q + (((size_t)b * N + rho / G) * a.Hq + kvh * G + rho % G) * D, D * 2);
            } else {
                const int kk = k - nq, row = t_lo + kk / 2;
                prefetch_l2_bulk(((kk & 1) ? a.v_new : a.k_new) + (((size_t)b * N + row) * a.Hkv + kvh) * D, D * 2);
            }
        }
    }

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool by_stagers = i >= kKFree0 && i <= kVReady1;
            const bool by_softmax = i == kPReady0 || i == kPReady1 || i == kSFree0 || i == kSFree1;
            const int count = i <= kRawV1 ? 32 : by_stagers ? kStageThreads : by_softmax ? kSoftWarps * 32 : 1;
            mbar_init(bars + i, count);
        }
        fence_mbar_init();
        *fail_s = 0;
    }
    if (warp == kMmaWarp) tc::alloc(tmem_slot, L::kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int st = tid - kStage0;  // stage thread index (valid for warps 4-7)
    uint8_t* rawK = smem + L::off_rawK;
    uint8_t* rawV = smem + L::off_rawV;
    auto issue_tile_raw = [&](int u, bool k_plane, bool v_plane) {
        const TileInfo ti = tile(u);
        if (k_plane)
            issue_raw<D, KT>(kq, a.ks, plane_row0, ti.start, ti.count, rawK + (u & 1) * FK::kRaw,
                               bars + kRawK0 + (u & 1), lane);
        if (v_plane)
            issue_raw<D, VT>(vq, a.vs, plane_row0, ti.start, ti.count, rawV + (u & 1) * FV::kRaw,
                               bars + kRawV0 + (u & 1), lane);
    };
    // the first two tiles' raw planes are requested at once
    if (warp == kLoadWarp || warp == kLoadWarp + 1)
        for (int u = 0; u < min(T, 2); ++u)
            if (!tile(u).tree) issue_tile_raw(u, warp == kLoadWarp, warp != kLoadWarp);

    // The stage warps go straight to their loop: they read only the raw
    // tiles (cached slots below P, or tree slots that the other warps
    // quantise and the load warps request after this block), so with early
    // prefetch they stage the first cached tiles before the dependency wait.
    // The other warps wait, prepare Q and quantise the tree rows, and meet at
    // their own barrier.
    const bool stage_warp = warp >= kSoftWarps && warp < kMmaWarp;
    const int pt = warp < kSoftWarps ? tid : tid - kStageThreads;  // index among the other warps
    if (early && !stage_warp) grid_dependency_wait();

    // ---- Q rows -> fp16 pairs in tensor memory: softmax thread r writes row
    //      r into its own lane (rows past the tile are zero); every load of a
    //      thread is issued before the first is used.  With a TQ3_0 cache the
    //      query goes into the keys' rotated basis first: the prep warps
    //      rotate the rows (one warp per row, fp32) into shared memory, half
    //      of the row tile at a time, and the softmax threads of that half
    //      copy their rows from there.
    const int pw = warp < kSoftWarps ? warp : warp - kStageWarps;  // prep warp index
    constexpr int kPrepWarps = kPrepThreads / 32;
    if constexpr (L::kRotated) {
        if (!stage_warp) {
            constexpr int QSS = D + 8;  // fp16 row stride (bank-conflict free row reads)
            __half* QS = reinterpret_cast<__half*>(smem + L::off_QS);
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                for (int rr = pw; rr < kRows / 2; rr += kPrepWarps) {
                    const int r = hf * (kRows / 2) + rr, rho = row0 + r;
                    float v[D / 32];
                    if (r < RT && rho < rows_valid) {
                        load_row_warp<D>(a.q + (((size_t)b * N + rho / G) * a.Hq + kvh * G + rho % G) * D, v, lane);
                        fwht_warp<D>(v, lane);
                    } else {
#pragma unroll
                        for (int j = 0; j < D / 32; ++j) v[j] = 0.f;
                    }
                    uint32_t hv[D / 64];
#pragma unroll
                    for (int j = 0; j < D / 64; ++j) hv[j] = pack_f16x2(v[2 * j], v[2 * j + 1]);
                    if constexpr (D / 64 == 4)
                        *reinterpret_cast<uint4*>(QS + rr * QSS + lane * (D / 32)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    else
                        *reinterpret_cast<uint2*>(QS + rr * QSS + lane * (D / 32)) = make_uint2(hv[0], hv[1]);
                }
                named_barrier_sync_n(kPrepBarrier, kPrepThreads);
                if (warp == 2 * hf || warp == 2 * hf + 1) {
                    const int rr = tid - hf * (kRows / 2);
                    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {  // 64 dims = 32 columns per store
                        uint32_t v[32];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 x = *reinterpret_cast<const uint4*>(QS + rr * QSS + c * 64 + j * 8);
                            v[4 * j] = x.x;
                            v[4 * j + 1] = x.y;
                            v[4 * j + 2] = x.z;
                            v[4 * j + 3] = x.w;
                        }
                        tc::st32u(tmem + lane_off + L::kQcol + (uint32_t)(c * 32), v);
                    }
                    tc::fence_before_sync();
                }
                named_barrier_sync_n(kPrepBarrier, kPrepThreads);  // the staging rows are free again
            }
        }
    } else if (warp < kSoftWarps) {
        const int r = tid, rho = row0 + r;
        const bool on = r < RT && rho < rows_valid;
        const uint4* src = on ? reinterpret_cast<const uint4*>(a.q + (((size_t)b * N + rho / G) * a.Hq + kvh * G + rho % G) * D)
                              : nullptr;
        constexpr int C8 = D / 8;  // 16-byte chunks of a row
        uint4 w[C8];
#pragma unroll
        for (int j = 0; j < C8; ++j) w[j] = on ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
#pragma unroll
        for (int c = 0; c < C8; c += 8) {  // 64 dims = 32 columns per store
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t x[4] = {w[c + j].x, w[c + j].y, w[c + j].z, w[c + j].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v[4 * j + e] = pack_f16x2(bf16_bits_to_float((uint16_t)(x[e] & 0xffff)),
                                              bf16_bits_to_float((uint16_t)(x[e] >> 16)));
            }
            tc::st32u(tmem + lane_off + L::kQcol + (uint32_t)(c * 4), v);
        }
        tc::fence_before_sync();
    }
    // ---- the tree's own keys and values: the CTA that attends to a tree
    //      tile quantises that tile's rows into the cache itself (every row
    //      tile's CTA writes the same bytes) and copies them back like a
    //      cached tile once this block's writes are visible
    if (!stage_warp) {
        const int r_lo = max(0, g0 - n_cache_tiles) * kTK;
        const int r_hi = min(n, (g0 + T - n_cache_tiles) * kTK);
        const int nblk = (r_hi > r_lo) ? (r_hi - r_lo) * NB : 0;
        if constexpr (L::kRotated) {
            // TQ3_0: each tree row is rotated as a whole before it is
            // quantised (one warp per row and plane)
            const int nrow = (r_hi > r_lo) ? r_hi - r_lo : 0;
            for (int k = pw; k < 2 * nrow; k += kPrepWarps) {
                const bool vplane = k & 1;
                const int row = r_lo + k / 2;
                float v[D / 32];
                load_row_warp<D>((vplane ? a.v_new : a.k_new) + (((size_t)b * N + row) * a.Hkv + kvh) * D, v, lane);
                fwht_warp<D>(v, lane);
                const size_t slot = plane_row0 + P + row;
                quantize_tq3_warp<D>(v, (vplane ? vq : kq) + slot * FK::KB, (vplane ? a.vs : a.ks) + slot * NB, lane);
            }
        }
        for (int k = pt; k < (L::kRotated ? 0 : 2 * nblk); k += kPrepThreads) {
            const bool vplane = k >= nblk;
            const int kk = vplane ? k - nblk : k, row = r_lo + kk / NB, blk = kk % NB;
            const uint16_t* src = (vplane ? a.v_new : a.k_new) + (((size_t)b * N + row) * a.Hkv + kvh) * D + blk * 32;
            const size_t slot = plane_row0 + P + row;
            if constexpr (!L::kRotated) {
                if (vplane)
                    quantize_block<VT>(src, vq + slot * FV::KB + blk * (FV::KB / NB), a.vs + slot * NB + blk);
                else
                    quantize_block<KT>(src, kq + slot * FK::KB + blk * (FK::KB / NB), a.ks + slot * NB + blk);
            }
        }
        __threadfence();
        fence_proxy_async_smem();
        asm volatile("fence.proxy.async.global;\n" ::: "memory");  // the tree rows are read back by bulk copies
        named_barrier_sync_n(kPrepBarrier, kPrepThreads);
    }

    const uint32_t tmem_O = tmem;  // columns [0, D)
    float m_run = -INFINITY, l_run = 0.f;

    if (warp < kSoftWarps) {
        // ================================================ softmax: thread = query row
        const int srow = tid;
        int lb = INT_MAX, rdepth = 0;
        uint64_t ramask = 0;
        {
            const int rho = row0 + srow;
            if (srow < RT && rho < rows_valid) {
                const int i = rho / G;
                rdepth = depth_s[i];
                ramask = amask_s[i];
                lb = (W > 0) ? P + depth_s[i] - W + 1 : INT_MIN;
            }
        }
        const float sl2 = a.scale * kLog2e;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        // a warp whose rows are all padding only keeps the barrier phases
        // in step (its P rows and O rows are never read back)
        const bool warp_active = 32 * warp < min(RT, rows_valid - row0);
        for (int t = 0; t < T && !warp_active; ++t) {
            const bool ok = __all_sync(0xffffffffu, wait_phase(bars + kSFull0 + (t & 1), (t >> 1) & 1));
            if (!ok) {
                if (lane == 0) atomicOr(fail_s, 1);
                break;
            }
            mbar_arrive(bars + kSFree0 + (t & 1));
            mbar_arrive(bars + kPReady0 + (t & 1));
        }
        for (int t = 0; t < T && warp_active; ++t) {
            const TileInfo ti = tile(t);
            bool ok = wait_phase(bars + kSFull0 + (t & 1), (t >> 1) & 1);
            ok = __all_sync(0xffffffffu, ok && !failed());
            if (!ok) {
                if (lane == 0) atomicOr(fail_s, 1);
                break;
            }
            tc::fence_after_sync();
            float s[kTK];
            {
                float sh[32], sl[32];
                tc::ld32(tmem + L::kScol + lane_off, sh);
                tc::ld32(tmem + L::kScol + lane_off + kTK, sl);
#pragma unroll
                for (int c = 0; c < kTK; ++c) s[c] = sh[c] + sl[c];
            }
            // the S buffer is read: the next tile's scores may go into it
            tc::fence_before_sync();
            mbar_arrive(bars + kSFree0 + (t & 1));
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (ti.tree) {
#pragma unroll
                for (int c = 0; c < kTK; ++c) {
                    const int l = ti.start - P + c;
                    const bool vis = c < ti.count && ((ramask >> l) & 1ull) && (W == 0 || depth_s[l] > rdepth - W);
                    s[c] = vis ? s[c] * sl2 : -INFINITY;
                    mx[c & 3] = fmaxf(mx[c & 3], s[c]);
                }
            } else {
                // visible: first <= c < lim (lb is INT_MIN without a window, INT_MAX for padding rows)
                const int lim = min(ti.count, kTK), first = (lb == INT_MIN) ? 0 : lb - ti.start;
#pragma unroll
                for (int c = 0; c < kTK; ++c) {
                    s[c] = (c < lim && c >= first) ? s[c] * sl2 : -INFINITY;
                    mx[c & 3] = fmaxf(mx[c & 3], s[c]);
                }
            }
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            float alpha = 1.f;
            bool rescale = false;
            if (mt > m_run + 8.f) {
                alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mt);
                m_run = mt;
                l_run *= alpha;
                rescale = t > 0;
            }
            if (__any_sync(0xffffffffu, rescale)) {
                // every product into O so far has completed before O is rescaled
                bool ok2 = __all_sync(0xffffffffu, wait_phase(bars + kODone0 + ((t - 1) & 1), ((t - 1) >> 1) & 1));
                if (!ok2) {
                    if (lane == 0) atomicOr(fail_s, 1);
                    break;
                }
                tc::fence_after_sync();
                const float al = rescale ? alpha : 1.f;
#pragma unroll 1
                for (int c0o = 0; c0o < D; c0o += 32) {
                    float o[32];
                    tc::ld32(tmem_O + lane_off + c0o, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= al;
                    tc::st32(tmem_O + lane_off + c0o, o);
                }
            }
            const float base = (m_run == -INFINITY) ? 0.f : m_run;
            uint32_t ph[kTK / 2], pl[kTK / 2];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < kTK; j += 2) {
                const float p0 = exp2f(s[j] - base), p1 = exp2f(s[j + 1] - base);
                ls[(j >> 1) & 3] += p0 + p1;
                const __half2 h2 = __floats2half2_rn(p0, p1);
                const float2 hf = __half22float2(h2);
                const __half2 l2 = __floats2half2_rn(p0 - hf.x, p1 - hf.y);
                ph[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
                pl[j / 2] = *reinterpret_cast<const uint32_t*>(&l2);
            }
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // P buffer t & 1 was last read by the products of tile t - 2
            if (t >= 2) {
                const bool okp = __all_sync(0xffffffffu, wait_phase(bars + kODone0 + (t & 1), ((t - 2) >> 1) & 1));
                if (!okp) {
                    if (lane == 0) atomicOr(fail_s, 1);
                    break;
                }
                tc::fence_after_sync();
            }
            // P_hi in the buffer's columns [0, kTK/2), P_lo in [kTK/2, kTK)
            const uint32_t tp = tmem + L::kPcol + (uint32_t)((t & 1) * kTK);
            tc::st16u(tp + lane_off, ph);
            tc::st16u(tp + lane_off + kTK / 2, pl);
            tc::fence_before_sync();
            mbar_arrive(bars + kPReady0 + (t & 1));
        }
        // the last PV
        if (__all_sync(0xffffffffu, T > 0 && !failed())) {
            bool ok = __all_sync(0xffffffffu, wait_phase(bars + kODone0 + ((T - 1) & 1), ((T - 1) >> 1) & 1));
            if (!ok && lane == 0) atomicOr(fail_s, 1);
            tc::fence_after_sync();
        }
    } else if (warp < kMmaWarp) {
        // ================================================ stage warps
        for (int t = 0; t <= T; ++t) {
            bool ok = true;
            if (t < T) {
                const TileInfo ti = tile(t);
                uint8_t* rk = rawK + (t & 1) * FK::kRaw;
                ok = ok && wait_phase(bars + kRawK0 + (t & 1), (t >> 1) & 1);
                const int shift = scale_shift<D, KT>(a.ks, plane_row0, ti.start);
                if (t >= 2) ok = ok && wait_phase(bars + kSFull0 + (t & 1), ((t - 2) >> 1) & 1);
                if (ok)
                    stage_hilo<D, KT>(rk, reinterpret_cast<const uint16_t*>(rk + FK::kRawCodes + shift), ti.count,
                                        smem + L::off_K + (t & 1) * L::kK,
                                        smem + L::off_K + (t & 1) * L::kK + L::kK / 2, st);
                mbar_arrive(bars + kKFree0 + (t & 1));  // raw K buffer of this parity released
                fence_proxy_async_smem();
                mbar_arrive(bars + kKReady0 + (t & 1));
            }
            if (t >= 1 && ok) {
                const int u = t - 1;
                const TileInfo tu = tile(u);
                uint8_t* rv = rawV + (u & 1) * FV::kRaw;
                ok = ok && wait_phase(bars + kRawV0 + (u & 1), (u >> 1) & 1);
                const int shift = scale_shift<D, VT>(a.vs, plane_row0, tu.start);
                // the products of tile u - 2 that read this V buffer have completed
                if (u >= 2) ok = ok && wait_phase(bars + kODone0 + (u & 1), ((u - 2) >> 1) & 1);
                unsigned char* vb = smem + L::off_V + (u & 1) * 2 * L::kV;
                if (ok)
                    stage_hilo<D, VT>(rv, reinterpret_cast<const uint16_t*>(rv + FV::kRawCodes + shift), tu.count,
                                        vb, vb + L::kV, st);
                mbar_arrive(bars + kVFree0 + (u & 1));  // raw V buffer of this parity released
                fence_proxy_async_smem();
                mbar_arrive(bars + kVReady0 + (u & 1));
            }
            // a failure is seen by every stage thread at the same iteration
            const bool bad = named_barrier_or(kStageBarrier, kStageThreads, !ok || failed());
            if (bad) {
                if (st == 0) atomicOr(fail_s, 1);
                break;
            }
        }
    } else if (warp == kLoadWarp || warp == kLoadWarp + 1) {
        // ================================================ raw tile copies: tile u
        // goes into buffer u & 1 once the stage warps have released tile u - 2.
        // One warp per plane, so a K request never waits behind a V buffer.
        const bool kside = warp == kLoadWarp;
        bool ok = true;
        asm volatile("fence.proxy.async.global;\n" ::: "memory");
        int issued = min(T, 2);  // tiles requested so far (the first two before the loop, tree tiles below)
        for (int u = 0; u < T && ok; ++u) {
            if (u < 2 && !tile(u).tree) continue;  // requested before the loop
            if (u >= 2) ok = wait_phase(bars + (kside ? kKFree0 : kVFree0) + (u & 1), ((u - 2) >> 1) & 1);
            if (ok) {
                issue_tile_raw(u, kside, !kside);
                issued = max(issued, u + 1);
            }
        }
        if (!__all_sync(0xffffffffu, ok) && lane == 0) atomicOr(fail_s, 1);
        // the last bulk copies into this plane's buffers have landed before
        // the CTA moves on (the stage warps have normally seen them already)
        for (int u = max(0, issued - 2); u < issued; ++u)
            wait_phase(bars + (kside ? kRawK0 : kRawV0) + (u & 1), (u >> 1) & 1);
    } else if (lane == 0) {
        // ================================================ MMA issue (one thread)
        constexpr uint32_t SBO = (D / 8) * 128;
        constexpr uint32_t idesc_qk = tc::idesc_f16(kRows, 2 * kTK, false);  // K_lo follows K_hi
        constexpr uint32_t idesc_pv = tc::idesc_f16(kRows, D, true);
        constexpr uint32_t V_LBO = (D / 8) * 128;
        // [S_hi | S_lo] of tile t = Q (tensor memory) [K_hi ; K_lo]^T
        auto issue_qk = [&](int t) {
            const uint32_t kb = smem_u32(smem + L::off_K + (t & 1) * L::kK);
            const uint32_t ts = tmem + L::kScol;
#pragma unroll 4
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_f16_ts(ts, tmem + L::kQcol + (uint32_t)(ks * 8), tc::smem_desc(kb + ks * 256, 128, SBO),
                               idesc_qk, ks > 0);
            tc::commit(bars + kSFull0 + (t & 1));
        };
        // Per tile t: the scores of tile t + 1 as soon as the softmax has
        // read those of tile t (one S buffer; P goes to its own buffers), so
        // they are formed while the softmax works; then the products of tile
        // t once its P is written.
        bool ok = T <= 0 || wait_phase(bars + kKReady0, 0);
        if (ok && T > 0) {
            tc::fence_after_sync();
            issue_qk(0);
        }
        for (int t = 0; t < T && ok; ++t) {
            if (t + 1 < T) {
                ok = wait_phase(bars + kKReady0 + ((t + 1) & 1), ((t + 1) >> 1) & 1) &&
                     wait_phase(bars + kSFree0 + (t & 1), (t >> 1) & 1);
                if (!ok) break;
                tc::fence_after_sync();
                issue_qk(t + 1);
            }
            ok = wait_phase(bars + kPReady0 + (t & 1), (t >> 1) & 1) &&
                 wait_phase(bars + kVReady0 + (t & 1), (t >> 1) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            // O += P_hi V_hi + P_hi V_lo + P_lo V_hi, P (tensor memory) in
            // buffer t & 1: P_hi in its columns [0, kTK/2), P_lo after
            const uint32_t ps = tmem + L::kPcol + (uint32_t)((t & 1) * kTK);
            const uint32_t vh = smem_u32(smem + L::off_V + (t & 1) * 2 * L::kV), vl = vh + (uint32_t)L::kV;
#pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks) {
                const uint64_t bh = tc::smem_desc(vh + ks * 2 * V_LBO, V_LBO, 128);
                const uint64_t bl = tc::smem_desc(vl + ks * 2 * V_LBO, V_LBO, 128);
                const uint32_t ah = ps + (uint32_t)(ks * 8), al = ps + (uint32_t)(kTK / 2 + ks * 8);
                tc::mma_f16_ts(tmem_O, ah, bh, idesc_pv, t > 0 || ks > 0);
                tc::mma_f16_ts(tmem_O, ah, bl, idesc_pv, true);
                tc::mma_f16_ts(tmem_O, al, bh, idesc_pv, true);
            }
            tc::commit(bars + kODone0 + (t & 1));
        }
        if (!ok) atomicOr(fail_s, 1);
        // every MMA issued above has completed before TMEM or smem is reused
        tc::commit(bars + kMmaFin);
        wait_phase(bars + kMmaFin, 0);
    }
    __syncthreads();
    const bool any_fail = failed();  // settled: every role has left its loop
    if (any_fail && tid == 0) raise_status(a.status, DFLV_DEV_TIMEOUT);
    // the next kernel may be scheduled while the partials are merged
    grid_launch_dependents();

    // ---- partial results to the CTA that finalises each row: rank q of the
    //      cluster owns rows q, q + CS, ...  Each row's partial is (O, max,
    //      sum), and one cluster barrier publishes them:
    //      * with a workspace, through global memory: each CTA, as soon as
    //        its loop ends, stages its rows' partials in its own shared
    //        memory (slot r: O in [0, D), max at D, sum at D + 1) and writes
    //        them to its block of the workspace with one bulk copy; the
    //        owners read their rows' partials back from the L2;
    //      * without one, into the owner's shared memory by posted cluster
    //        stores, once every CTA has left its tile loop (the receiving
    //        region reuses the tile buffers).  Slot (s, q) of an owner holds
    //        peer q's partial of its s-th row.
    float* Rcv = reinterpret_cast<float*>(smem + L::off_Om);
    const bool gmerge = a.ws != nullptr;  // uniform over the launch
    float* wsb = gmerge ? reinterpret_cast<float*>(a.ws) +
                              (((size_t)b * a.Hkv + kvh) * (gridDim.y / a.Hkv) + rt) * CS * RT * OS
                        : nullptr;
    const int rows_here = min(RT, rows_valid - row0);  // rows 0 .. rows_here-1 are valid
    const bool have_o = T > 0 && !any_fail;  // uniform over the CTA
    if (gmerge) {
        // Staged row-major in this CTA's shared memory (slot r: O in
        // [0, D), max at D, sum at D + 1) by eight warps -- the softmax
        // warps take O's first D/2 columns, the stage warps the same TMEM
        // lanes' other half -- then written out by one bulk copy per 32-row
        // quarter, issued by four threads at once.
        if (warp < kMmaWarp) {
            const int r = (warp & 3) * 32 + lane;
            const bool valid = r < rows_here;
            bool ok_o = have_o;
            if (have_o && warp >= kSoftWarps) {
                // the stage warps have not seen the last products complete
                ok_o = __all_sync(0xffffffffu,
                                  wait_phase(bars + kODone0 + ((T - 1) & 1), ((T - 1) >> 1) & 1));
                tc::fence_after_sync();
            }
            if (ok_o) {
                // the TMEM loads are warp-collective: every lane loads, only
                // the lanes of valid rows store
                const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
                const int cb = warp < kSoftWarps ? 0 : D / 2;
#pragma unroll 1
                for (int c0o = cb; c0o < cb + D / 2; c0o += 32) {
                    float o[32];
                    tc::ld32(tmem_O + lane_off + c0o, o);
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(Rcv + (size_t)r * OS + c0o + e) =
                                make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                    }
                }
            } else if (have_o && lane == 0) {
                raise_status(a.status, DFLV_DEV_TIMEOUT);  // this CTA's O is not staged
            }
            if (warp < kSoftWarps && valid)
                *reinterpret_cast<float2*>(Rcv + (size_t)r * OS + D) =
                    make_float2(have_o ? m_run : -INFINITY, have_o ? l_run : 0.f);
            fence_proxy_async_smem();  // the staged rows go out through the bulk-copy engine
        }
    } else {
        // into the owners' shared memory (the tile buffers), once every CTA
        // has left its loop
        cluster_sync_all();
        if (warp < kSoftWarps) {
            const int r = tid;
            const bool valid = r < rows_here;
            const int owner = valid ? r % CS : 0, slot = valid ? r / CS : 0;
            const uint32_t dst = map_to_rank(smem_u32(Rcv + (size_t)(slot * CS + rank) * OS), (uint32_t)owner);
            if (have_o) {
                const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
                for (int c0o = 0; c0o < D; c0o += 64) {
                    uint32_t o[2][32];  // two loads in flight before one wait
                    tc::ld32_nowait(tmem_O + lane_off + c0o, o[0]);
                    tc::ld32_nowait(tmem_O + lane_off + c0o + 32, o[1]);
                    tc::wait_ld();
                    if (valid) {
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                            for (int e = 0; e < 32; e += 4)
                                st_dsmem_f4(dst + (uint32_t)(c0o + 32 * h2 + e) * 4, __uint_as_float(o[h2][e]),
                                            __uint_as_float(o[h2][e + 1]), __uint_as_float(o[h2][e + 2]),
                                            __uint_as_float(o[h2][e + 3]));
                    }
                }
            }
            if (valid) st_dsmem_f2(dst + (uint32_t)D * 4, have_o ? m_run : -INFINITY, have_o ? l_run : 0.f);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::dealloc(tmem, L::kTmemCols);
    }
    if (gmerge && lane == 0 && warp < kSoftWarps && 32 * warp < rows_here) {
        const int nr = min(32, rows_here - 32 * warp);
        bulk_s2g(wsb + ((size_t)rank * RT + 32 * warp) * OS, Rcv + (size_t)32 * warp * OS, (uint32_t)(nr * OS * 4));
        bulk_s2g_wait();
    }
    cluster_sync_all();  // every partial is visible to its owner

    // ---- merge the owned rows
    constexpr int nwarps = kThreads / 32;
    constexpr int PL = D / 32;  // output floats per lane when a warp takes a whole row
    if (gmerge && L::kRotated) {
        // TQ3_0: the output is rotated back after the merge, which needs a
        // whole row in one warp: one warp per owned row, peers in batches
        // of eight (every load of a batch in flight at once), merged online
        const int n_own = (rank < rows_here) ? (rows_here - 1 - rank) / CS + 1 : 0;
        for (int slot = warp; slot < n_own; slot += nwarps) {
            const int r = rank + slot * CS, rho = row0 + r;
            float Mr = -INFINITY, Lt = 0.f, acc[PL];
#pragma unroll
            for (int e = 0; e < PL; ++e) acc[e] = 0.f;
            for (int q0 = 0; q0 < CS; q0 += 8) {
                float2 ml[8];
                float ov[8][PL];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    ml[q] = make_float2(-INFINITY, 0.f);
#pragma unroll
                    for (int e = 0; e < PL; ++e) ov[q][e] = 0.f;
                    if (q0 + q < CS) {
                        const float* src = wsb + ((size_t)(q0 + q) * RT + r) * OS;
                        ml[q] = __ldcg(reinterpret_cast<const float2*>(src + D));
#pragma unroll
                        for (int e = 0; e < PL; e += 4) {
                            const float4 x = __ldcg(reinterpret_cast<const float4*>(src + lane * PL + e));
                            ov[q][e] = x.x;
                            ov[q][e + 1] = x.y;
                            ov[q][e + 2] = x.z;
                            ov[q][e + 3] = x.w;
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float mq = ml[q].x;
                    if (mq == -INFINITY) continue;  // absent peer, or one without keys for this row
                    if (mq > Mr) {
                        const float sc = (Mr == -INFINITY) ? 0.f : exp2f(Mr - mq);
                        Lt *= sc;
#pragma unroll
                        for (int e = 0; e < PL; ++e) acc[e] *= sc;
                        Mr = mq;
                    }
                    const float w = exp2f(mq - Mr);
                    Lt = fmaf(w, ml[q].y, Lt);
#pragma unroll
                    for (int e = 0; e < PL; ++e) acc[e] = fmaf(w, ov[q][e], acc[e]);
                }
            }
            const float inv = 1.f / Lt;
#pragma unroll
            for (int e = 0; e < PL; ++e) acc[e] *= inv;
            fwht_warp<D>(acc, lane);  // back from the values' rotated basis
            const int i = rho / G, gh = rho % G;
            float* dsto = a.out + (((size_t)b * N + i) * a.Hq + kvh * G + gh) * D + lane * PL;
#pragma unroll
            for (int e = 0; e < PL; e += 4)
                *reinterpret_cast<float4*>(dsto + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
        }
        return;
    }
    if (gmerge) {
        // The row tile's outputs are cut into items of four consecutive
        // floats of a row, and the cluster's CTAs take consecutive ranges
        // of them (one item per thread at the usual shapes), so every CTA
        // merges about the same amount and each thread issues all of its
        // peers' loads at once: one round trip to the L2.  Peers are merged
        // in rank order.
        constexpr int NCH = D / 4;
        const int items = rows_here * NCH;
        const int per = (items + CS - 1) / CS;
        const int it0 = rank * per, it1 = min(items, it0 + per);
        for (int item = it0 + tid; item < it1; item += kThreads) {
            const int r = item / NCH, c0 = (item % NCH) * 4, rho = row0 + r;
            float2 ml[16];
            float4 ov[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                ml[q] = make_float2(-INFINITY, 0.f);
                ov[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q < CS) {
                    const float* src = wsb + ((size_t)q * RT + r) * OS;
                    ov[q] = __ldcg(reinterpret_cast<const float4*>(src + c0));
                    ml[q] = __ldcg(reinterpret_cast<const float2*>(src + D));
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < 16; ++q) M = fmaxf(M, ml[q].x);
            const float bse = (M == -INFINITY) ? 0.f : M;
            float Lt = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                // absent peers and peers without keys for this row: max -inf, weight 0
                const float w = (ml[q].x == -INFINITY) ? 0.f : exp2f(ml[q].x - bse);
                Lt = fmaf(w, ml[q].y, Lt);
                if (w != 0.f) {
                    acc[0] = fmaf(w, ov[q].x, acc[0]);
                    acc[1] = fmaf(w, ov[q].y, acc[1]);
                    acc[2] = fmaf(w, ov[q].z, acc[2]);
                    acc[3] = fmaf(w, ov[q].w, acc[3]);
                }
            }
            const float inv = 1.f / Lt;
            const int i = rho / G, gh = rho % G;
            float* dsto = a.out + (((size_t)b * N + i) * a.Hq + kvh * G + gh) * D + c0;
            *reinterpret_cast<float4*>(dsto) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
        }
        return;
    }
    // one warp per row, from local shared memory
    for (int slot = warp; rank + slot * CS < RT; slot += nwarps) {
        const int r = rank + slot * CS, rho = row0 + r;
        if (rho >= rows_valid) continue;
        float Lt = 0.f, acc[PL];
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] = 0.f;
        const float* base = Rcv + (size_t)slot * CS * OS;
        float M = -INFINITY;
        for (int q = 0; q < CS; ++q) M = fmaxf(M, base[q * OS + D]);
        const float bse = (M == -INFINITY) ? 0.f : M;
        for (int q = 0; q < CS; ++q) {
            const float mq = base[q * OS + D];
            if (mq == -INFINITY) continue;  // a peer without keys for this row sent no O
            const float w = exp2f(mq - bse);
            Lt = fmaf(w, base[q * OS + D + 1], Lt);
            const float* oq = base + q * OS + lane * PL;
#pragma unroll
            for (int e = 0; e < PL; e += 4) {
                const float4 x = *reinterpret_cast<const float4*>(oq + e);
                acc[e] = fmaf(w, x.x, acc[e]);
                acc[e + 1] = fmaf(w, x.y, acc[e + 1]);
                acc[e + 2] = fmaf(w, x.z, acc[e + 2]);
                acc[e + 3] = fmaf(w, x.w, acc[e + 3]);
            }
        }
        const float inv = 1.f / Lt;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] *= inv;
        if constexpr (L::kRotated) fwht_warp<D>(acc, lane);  // back from the values' rotated basis
        const int i = rho / G, gh = rho % G;
        float* dst = a.out + (((size_t)b * N + i) * a.Hq + kvh * G + gh) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
    }
}

// How many clusters of cs CTAs of this kernel can be resident at once at
// this shared-memory size (queried once per kernel instantiation and
// cluster size; sizes above 8 are the non-portable ones, allowed here for
// the kernel before the query and so before any launch that uses them).
template <int D, int KT, int VT>
int active_clusters(int cs) {
    static int cache[17] = {0};  // one table per instantiation
    if (cs < 1 || cs > 16) return 0;
    if (cache[cs] == 0) {
        auto kern = attn_tc_kernel<D, KT, VT>;
        int n = 0;
        if (cs > 8) cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = TcLayout<D, KT, VT>::total;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        cudaGetLastError();
        cache[cs] = n > 0 ? n : -1;
    }
    return cache[cs] > 0 ? cache[cs] : 0;
}

struct TcPlan {
    int n_rt, RT, CS;
};

// Row tiles and cluster size of a launch (the device's cluster occupancy
// enters, so the plan is per device).
template <int D, int KT, int VT>
TcPlan plan_tc(const AttnVerifyArgs& a) {
    const int rows = (a.Hq / a.Hkv) * a.N_max;
    const long range = (a.window > 0) ? (long)a.window - 1 : (long)a.cap;
    const long tiles = (range + kTK - 1) / kTK + 3;
    // Cluster size and row tiles by a small cost model: a CTA costs its share
    // of the key tiles plus a fixed prologue-and-merge overhead (in tile
    // units), and the launch costs that times the number of waves of
    // clusters the GPU can hold at once (the occupancy query).  Any size up
    // to 16 is allowed (the key tiles split by cost, so sizes between powers
    // of two also shorten the longest CTA).  Short key ranges end up with one
    // wave of the largest resident clusters; long ranges with several waves
    // of smaller ones, which keeps every SM busy.
    constexpr double kOverheadTiles = 3.0;
    auto est = [&](int n_rt, int cs) {
        const long clusters = (long)n_rt * a.Hkv * a.B;
        const int act = active_clusters<D, KT, VT>(cs);
        if (act <= 0) return 1e30;
        const long waves = (clusters + act - 1) / act;
        return (double)waves * ((double)tiles / cs + kOverheadTiles);
    };
    auto choose_cs = [&](int n_rt, double& best) {
        int bcs = 1;
        best = est(n_rt, 1);
        for (int cs = 2; cs <= 16 && cs * 2 <= tiles; ++cs) {
            const double e = est(n_rt, cs);
            if (e < best) {
                best = e;
                bcs = cs;
            }
        }
        return bcs;
    };
    // row tiles: as few as the 128-row MMA allows, or one more (rows of at
    // least 32 each) when that is cheaper by the same model
    int n_rt = (rows + kRows - 1) / kRows;
    double e1, e2;
    int cs = choose_cs(n_rt, e1);
    {
        const int n2 = n_rt + 1;
        if ((rows + n2 - 1) / n2 >= 32) {
            const int cs2 = choose_cs(n2, e2);
            if (e2 < e1) {
                n_rt = n2;
                cs = cs2;
            }
        }
    }
    return TcPlan{n_rt, (rows + n_rt - 1) / n_rt, cs};
}

// Workspace of the global merge: one partial row (O, max, sum, two words
// of padding) per (sequence, KV head, row tile, cluster rank, row).
template <int D, int KT, int VT>
size_t ws_bytes_tc(const AttnVerifyArgs& a) {
    // the occupancy query behind the plan needs the kernel's shared-memory
    // size granted first
    if (ensure_smem(attn_tc_kernel<D, KT, VT>, TcLayout<D, KT, VT>::total) != cudaSuccess) return 0;
    const TcPlan p = plan_tc<D, KT, VT>(a);
    return (size_t)a.B * a.Hkv * p.n_rt * p.CS * p.RT * (D + 4) * sizeof(float);
}

template <int D, int KT, int VT>
cudaError_t launch_tc(const AttnVerifyArgs& a, cudaStream_t stream) {
    using L = TcLayout<D, KT, VT>;
    auto kern = attn_tc_kernel<D, KT, VT>;
    cudaError_t e = ensure_smem(kern, L::total);
    if (e != cudaSuccess) return e;
    const TcPlan p = plan_tc<D, KT, VT>(a);
    AttnVerifyArgs b = a;
    if (!b.ws || b.ws_bytes < (size_t)a.B * a.Hkv * p.n_rt * p.CS * p.RT * (D + 4) * sizeof(float)) b.ws = nullptr;
    b.flags &= ~kFlagPrefetchInputs;
    if ((a.flags & DFLV_FLAG_EARLY_PREFETCH) && (long)p.n_rt * a.Hkv * a.B <= active_clusters<D, KT, VT>(p.CS))
        b.flags |= kFlagPrefetchInputs;
    return launch_pdl(kern, dim3(p.CS, p.n_rt * a.Hkv, a.B), dim3(kThreads), L::total, stream, p.CS, b, p.RT, p.CS);
}

}  // namespace

template <int D>
cudaError_t launch_tc_d(const AttnVerifyArgs& a, cudaStream_t stream) {
    constexpr int Q8 = DFLV_KV_Q8_0, Q4 = DFLV_KV_Q4_0;
    switch (a.type) {
        case DFLV_KV_Q8_0: return launch_tc<D, Q8, Q8>(a, stream);
        case DFLV_KV_Q4_0: return launch_tc<D, Q4, Q4>(a, stream);
        case DFLV_KV_Q8_0_Q4_0: return launch_tc<D, Q8, Q4>(a, stream);
        case DFLV_KV_Q4_0_Q8_0: return launch_tc<D, Q4, Q8>(a, stream);
        case DFLV_KV_TQ3_0: return launch_tc<D, DFLV_KV_TQ3_0, DFLV_KV_TQ3_0>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attn_tree_verify_tc(const AttnVerifyArgs& a, cudaStream_t stream) {
    switch (a.D) {
        case 128: return launch_tc_d<128>(a, stream);
        case 256: return launch_tc_d<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
size_t ws_bytes_tc_d(const AttnVerifyArgs& a) {
    constexpr int Q8 = DFLV_KV_Q8_0, Q4 = DFLV_KV_Q4_0;
    switch (a.type) {
        case DFLV_KV_Q8_0: return ws_bytes_tc<D, Q8, Q8>(a);
        case DFLV_KV_Q4_0: return ws_bytes_tc<D, Q4, Q4>(a);
        case DFLV_KV_Q8_0_Q4_0: return ws_bytes_tc<D, Q8, Q4>(a);
        case DFLV_KV_Q4_0_Q8_0: return ws_bytes_tc<D, Q4, Q8>(a);
        case DFLV_KV_TQ3_0: return ws_bytes_tc<D, DFLV_KV_TQ3_0, DFLV_KV_TQ3_0>(a);
        default: return 0;
    }
}

size_t attn_workspace_bytes_tc(const AttnVerifyArgs& a) {
    switch (a.D) {
        case 128: return ws_bytes_tc_d<128>(a);
        case 256: return ws_bytes_tc_d<256>(a);
        default: return 0;
    }
}

}  // namespace dflv
