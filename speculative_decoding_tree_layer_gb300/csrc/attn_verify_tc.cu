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
// query rows); the cluster's CTAs split the visible keys (and the tree
// block) into 32-key tiles.  Per CTA and tile:
//   * the int8 / 4-bit codes arrive by 16-byte cp.async (double-buffered)
//     and are staged as a pair of fp16 tiles hi + lo with the block scale
//     folded in (d * code is exact in fp32; hi = fp16(x), lo = fp16(x - hi)),
//     so the products below are exact to ~2^-22;
//   * one thread issues tcgen05.mma: [S_hi | S_lo] = Q [K_hi ; K_lo]^T into
//     tensor memory (M = 128 rows, N = 64 = the two 32-key halves stored
//     back to back, K = head size); S = S_hi + S_lo;
//   * eight warps read S (TMEM lane = query row; warps w and w + 4 share a
//     lane range and take 16 keys each), apply the tree / window mask, run an
//     fp32 online softmax with a lazily updated running max (rescaling O in
//     tensor memory only when a row's max grows by more than 2^8), and write
//     P as fp16 hi + lo;
//   * one thread issues O += P_hi V_hi + P_hi V_lo + P_lo V_hi (M = 128,
//     N = head size, K = 32) with O resident in tensor memory across tiles;
//   * partial (max, sum, O) are merged across the cluster through
//     distributed shared memory.
// Operands use the no-swizzle core-matrix layout described in tcgen05.cuh.
#include <climits>

#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "tree.cuh"

namespace dflv {

namespace {

using namespace attn;

constexpr int kTK = 32;        // keys per tile
constexpr int kRows = 128;     // MMA M: query rows per CTA
constexpr int kThreads = 256;  // all warps stage; softmax: two threads per row (16 keys each)

template <int D, int TYPE>
struct TcSmem {
    static constexpr int NB = D / 32;
    static constexpr int KB = (TYPE == DFLV_KV_Q8_0) ? D : D / 2;  // code bytes per key row
    static constexpr int RSK = KB + 16;                               // padded raw row stride
    static constexpr int OS = D + 4;                                  // merge row stride (floats)
    static constexpr size_t kHeader = 3072;  // tree arrays, barriers, [2][128] exchange floats at 2048
    static constexpr size_t kQ = (size_t)kRows * D * 2;
    static constexpr size_t kKV = (size_t)kTK * D * 2;   // one of K_hi, K_lo, V_hi, V_lo
    static constexpr size_t kP = (size_t)kRows * kTK * 2;
    static constexpr size_t kRawCodes = (size_t)kTK * RSK;
    static constexpr size_t kRawScales = (size_t)kTK * NB * 2;
    static constexpr size_t kRaw = 2 * kRawCodes + 2 * kRawScales;
    static constexpr size_t off_Q = kHeader;
    static constexpr size_t off_Khi = off_Q + kQ;
    static constexpr size_t off_Klo = off_Khi + kKV;
    static constexpr size_t off_Vhi = off_Klo + kKV;
    static constexpr size_t off_Vlo = off_Vhi + kKV;
    static constexpr size_t off_Phi = off_Vlo + kKV;
    static constexpr size_t off_Plo = off_Phi + kP;
    static constexpr size_t off_raw = off_Plo + kP;
    static constexpr size_t loop_total = off_raw + 2 * kRaw;
    static constexpr size_t off_Om = kHeader;
    static constexpr size_t off_Mm = off_Om + (size_t)kRows * OS * 4;
    static constexpr size_t off_Lm = off_Mm + (size_t)kRows * 4;
    static constexpr size_t merge_total = off_Lm + (size_t)kRows * 4;
    static constexpr size_t total = loop_total > merge_total ? loop_total : merge_total;
    static constexpr uint32_t kTmemCols = (D + 2 * kTK <= 256) ? 256 : 512;  // O at column 0, S after it
};

// Stage one 32-key tile of K or V codes as fp16 hi + lo with the block scale
// folded in; rows past count are zero.  Items are ordered key % 8 fastest so
// that 8 consecutive threads fill one 128-byte run of a core matrix.
template <int D, int TYPE>
DFLV_DEVINL void stage_hilo(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int count,
                            uint8_t* __restrict__ hi, uint8_t* __restrict__ lo, int tid) {
    using S = TcSmem<D, TYPE>;
    constexpr int C8 = D / 8;
    for (int idx = tid; idx < kTK * C8; idx += kThreads) {
        const int c = (idx & 7) + (idx / (8 * C8)) * 8;  // key
        const int d8 = (idx >> 3) % C8;                    // 8-dim chunk
        uint4 h = make_uint4(0, 0, 0, 0), l = make_uint4(0, 0, 0, 0);
        if (c < count) {
            const float sc = __half2float(__ushort_as_half(scales[c * S::NB + (d8 * 8) / 32]));
            float x[8];
            if constexpr (TYPE == DFLV_KV_Q8_0) {
                const uint2 w = *reinterpret_cast<const uint2*>(codes + c * S::RSK + d8 * 8);
                const uint32_t ww[2] = {w.x, w.y};
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = sc * (float)(int8_t)((ww[e >> 2] >> (8 * (e & 3))) & 0xff);
            } else {
                const int blk = (d8 * 8) / 32, off = (d8 * 8) % 32;
                const uint2 w = *reinterpret_cast<const uint2*>(codes + c * S::RSK + blk * 16 + (off & 15));
                const uint32_t ww[2] = {w.x, w.y};
                const int sh = off >= 16 ? 4 : 0;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    x[e] = sc * (float)((int)((ww[e >> 2] >> (8 * (e & 3) + sh)) & 15) - 8);
            }
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __half2 h2 = __floats2half2_rn(x[2 * e], x[2 * e + 1]);
                const float2 hf = __half22float2(h2);
                const __half2 l2 = __floats2half2_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
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

DFLV_DEVINL bool wait_phase(uint64_t* bar, uint32_t parity) {
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

template <int D, int TYPE>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnVerifyArgs a, int RT, int CS) {
    using S = TcSmem<D, TYPE>;
    constexpr int NB = S::NB, KB = S::KB, RSK = S::RSK, OS = S::OS;
    extern __shared__ __align__(1024) unsigned char smem[];
    int32_t* par_s = reinterpret_cast<int32_t*>(smem);
    int32_t* depth_s = par_s + kMaxNodes;
    uint64_t* amask_s = reinterpret_cast<uint64_t*>(smem + 512);
    uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + 1024);   // QK done
    uint64_t* bar_o = bar_s + 1;                                   // PV done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 1040);
    int32_t* fail_s = reinterpret_cast<int32_t*>(smem + 1044);
    float* xch_s = reinterpret_cast<float*>(smem + 2048);  // [2][128] per-half tile max / row sum
    unsigned char* Q_s = smem + S::off_Q;
    unsigned char* Khi_s = smem + S::off_Khi;
    unsigned char* Klo_s = smem + S::off_Klo;
    unsigned char* Vhi_s = smem + S::off_Vhi;
    unsigned char* Vlo_s = smem + S::off_Vlo;
    unsigned char* Phi_s = smem + S::off_Phi;
    unsigned char* Plo_s = smem + S::off_Plo;
    unsigned char* raw_s = smem + S::off_raw;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int kvh = blockIdx.y % a.Hkv, rt = blockIdx.y / a.Hkv, b = blockIdx.z;
    const int G = a.Hq / a.Hkv, N = a.N_max, W = a.window;

    grid_dependency_wait();
    grid_launch_dependents();
    const int n = __ldg(a.n_nodes + b), P = __ldg(a.n_past + b);
    // Uniform over the cluster: every CTA leaves before any cluster barrier.
    if (P < 0 || P + n > a.cap || n < 1 || n > N) {
        if (tid == 0 && rank == 0 && rt == 0 && kvh == 0)
            raise_status(a.status, (n < 1 || n > N) ? DFLV_DEV_TOPOLOGY : DFLV_DEV_CAPACITY);
        return;
    }
    const int rows_valid = G * n, row0 = rt * RT;
    if (row0 >= rows_valid) return;

    const size_t plane_row0 = ((size_t)b * a.Hkv + kvh) * a.cap;
    uint8_t* kq = reinterpret_cast<uint8_t*>(a.kq);
    uint8_t* vq = reinterpret_cast<uint8_t*>(a.vq);

    // tiles: cache keys [lo, P) then the tree slots [P, P + n), 32 keys each
    const int lo = (W > 0) ? max(0, P - W + 1) : 0;
    const int n_cache_tiles = (P - lo + kTK - 1) / kTK;
    const int n_tiles = n_cache_tiles + (n + kTK - 1) / kTK;
    auto tile_start = [&](int t) { return t < n_cache_tiles ? lo + t * kTK : P + (t - n_cache_tiles) * kTK; };
    auto tile_count = [&](int t) {
        return t < n_cache_tiles ? min(kTK, P - (lo + t * kTK)) : min(kTK, n - (t - n_cache_tiles) * kTK);
    };
    auto issue_tile = [&](int t, int buf) {
        const int start = tile_start(t), count = tile_count(t);
        uint8_t* base = raw_s + buf * S::kRaw;
        constexpr int CPR = KB / 16;
        for (int idx = tid; idx < count * CPR; idx += kThreads) {
            const int c = idx / CPR, ch = idx % CPR;
            const size_t g = (plane_row0 + start + c) * KB + ch * 16;
            cp_async16(base + c * RSK + ch * 16, kq + g);
            cp_async16(base + S::kRawCodes + c * RSK + ch * 16, vq + g);
        }
        uint8_t* ksd = base + 2 * S::kRawCodes;
        uint8_t* vsd = ksd + S::kRawScales;
        for (int c = tid; c < count; c += kThreads) {
            const size_t g = (plane_row0 + start + c) * NB;
            if constexpr (NB * 2 == 16) {
                cp_async16(ksd + c * 16, a.ks + g);
                cp_async16(vsd + c * 16, a.vs + g);
            } else {
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(ksd + c * 8)), "l"(a.ks + g) : "memory");
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(vsd + c * 8)), "l"(a.vs + g) : "memory");
            }
        }
        cp_async_commit();
    };

    // ---- set-up: TMEM, barriers, first tile, tree quantisation, topology
    if (warp == 0) tc::alloc(tmem_slot, S::kTmemCols);
    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
        *fail_s = 0;
    }
    int t_cur = rank;
    if (t_cur < n_cache_tiles) issue_tile(t_cur, 0);
    {
        const int mine = (n > rank) ? (n - rank + CS - 1) / CS : 0;
        for (int item = tid; item < mine * 2 * NB; item += kThreads) {
            const int j = item / (2 * NB), which = (item / NB) % 2, blk = item % NB;
            const int row = rank + CS * j;
            const uint16_t* src = (which ? a.v_new : a.k_new) + (((size_t)b * N + row) * a.Hkv + kvh) * D + blk * 32;
            const size_t slot = plane_row0 + P + row;
            quantize_block<TYPE>(src, (which ? vq : kq) + slot * KB + blk * (KB / NB),
                                 (which ? a.vs : a.ks) + slot * NB + blk);
        }
    }
    const bool topo_ok = block_tree_topology(a.parent + (size_t)b * N, n, N, par_s, depth_s, amask_s,
                                             (rank == 0 && rt == 0 && kvh == 0) ? a.status : nullptr);
    if (!topo_ok) {  // uniform over the cluster: the parent array is shared
        cp_async_wait<0>();
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::dealloc(*tmem_slot, S::kTmemCols);
        return;
    }
    __threadfence();
    cluster_sync_all();  // tree slots written by the whole cluster are visible
    if (t_cur >= n_cache_tiles) {
        if (t_cur < n_tiles) issue_tile(t_cur, 0);
        else cp_async_commit();
    }

    // ---- Q rows -> fp16, core-matrix layout (rows past the tile are zero)
    {
        // all of this thread's loads first (kRows * D / 8 / kThreads of them),
        // then the conversions and stores
        constexpr int C8 = D / 8;
        constexpr int PER = kRows * C8 / kThreads;
        uint4 inv[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = tid + j * kThreads;
            const int r = (idx & 7) + (idx / (8 * C8)) * 8;
            const int d8 = (idx >> 3) % C8;
            const int rho = row0 + r;
            inv[j] = make_uint4(0, 0, 0, 0);
            if (r < RT && rho < rows_valid) {
                const int i = rho / G, gh = rho % G;
                inv[j] = __ldg(reinterpret_cast<const uint4*>(
                    a.q + (((size_t)b * N + i) * a.Hq + kvh * G + gh) * D + d8 * 8));
            }
        }
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = tid + j * kThreads;
            const int r = (idx & 7) + (idx / (8 * C8)) * 8;
            const int d8 = (idx >> 3) % C8;
            const uint32_t w[4] = {inv[j].x, inv[j].y, inv[j].z, inv[j].w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = pack_f16x2(bf16_bits_to_float((uint16_t)(w[e] & 0xffff)),
                                  bf16_bits_to_float((uint16_t)(w[e] >> 16)));
            *reinterpret_cast<uint4*>(Q_s + tc::cm_offset(r, d8 * 8, D)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }

    // ---- per-row state: thread tid owns row tid % 128, key half tid / 128
    const int srow = tid & (kRows - 1), half = tid >> 7;
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
    float m_run = -INFINITY, l_run = 0.f;

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_O = tmem;          // columns [0, D)
    const uint32_t tmem_S = tmem + D;      // columns [D, D + 64): Q.K_hi then Q.K_lo
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // warps w and w+4 share lanes

    constexpr uint32_t idesc_qk = tc::idesc_f16(kRows, 2 * kTK, false);  // K_lo follows K_hi in smem
    constexpr uint32_t idesc_pv = tc::idesc_f16(kRows, D, true);
    uint32_t phase = 0;
    bool o_valid = false;
    int buf = 0;
    for (; t_cur < n_tiles; t_cur += CS, buf ^= 1) {
        const int t_next = t_cur + CS;
        if (t_next < n_tiles) issue_tile(t_next, buf ^ 1);
        else cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const bool tree_tile = t_cur >= n_cache_tiles;
        const int start = tile_start(t_cur), count = tile_count(t_cur);
        const uint8_t* rb = raw_s + buf * S::kRaw;
        const uint16_t* ksb = reinterpret_cast<const uint16_t*>(rb + 2 * S::kRawCodes);
        const uint16_t* vsb = reinterpret_cast<const uint16_t*>(rb + 2 * S::kRawCodes + S::kRawScales);
        stage_hilo<D, TYPE>(rb, ksb, count, Khi_s, Klo_s, tid);
        stage_hilo<D, TYPE>(rb + S::kRawCodes, vsb, count, Vhi_s, Vlo_s, tid);
        fence_proxy_async_smem();
        __syncthreads();

        // [S_hi | S_lo] = Q [K_hi ; K_lo]^T
        if (tid == 0 && !*fail_s) {
            tc::fence_after_sync();
            const uint32_t qa = smem_u32(Q_s), kh = smem_u32(Khi_s);
            constexpr uint32_t SBO = (D / 8) * 128;
#pragma unroll 4
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_f16(tmem_S, tc::smem_desc(qa + ks * 256, 128, SBO), tc::smem_desc(kh + ks * 256, 128, SBO),
                            idesc_qk, ks > 0);
            tc::commit(bar_s);
        }

        {
            // warp-uniform: the tcgen05 loads below are .sync.aligned
            const bool ok = __all_sync(0xffffffffu, *fail_s == 0 && wait_phase(bar_s, phase));
            if (!ok && lane == 0) atomicOr(fail_s, 1);
            tc::fence_after_sync();
            constexpr int HK = kTK / 2;  // keys per thread
            float s[HK];
            if (ok) {
                float sh[32], sl[32];
                tc::ld32(tmem_S + lane_off, sh);
                tc::ld32(tmem_S + lane_off + kTK, sl);
#pragma unroll
                for (int c = 0; c < HK; ++c) s[c] = half ? sh[HK + c] + sl[HK + c] : sh[c] + sl[c];
            }
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < HK; ++j) {
                const int c = half * HK + j;
                bool vis;
                if (tree_tile) {
                    const int l = start - P + c;
                    vis = c < count && ((ramask >> l) & 1ull) && (W == 0 || depth_s[l] > rdepth - W);
                } else {
                    vis = c < count && start + c >= lb;
                }
                s[j] = (vis && ok) ? s[j] * sl2 : -INFINITY;
                mt = fmaxf(mt, s[j]);
            }
            xch_s[half * kRows + srow] = mt;
            __syncthreads();
            mt = fmaxf(mt, xch_s[(half ^ 1) * kRows + srow]);
            float alpha = 1.f;
            bool rescale = false;
            if (mt > m_run + 8.f) {
                alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mt);
                m_run = mt;
                l_run *= alpha;
                rescale = o_valid;
            }
            const float base = (m_run == -INFINITY) ? 0.f : m_run;
            uint32_t ph[HK / 2], pl[HK / 2];
#pragma unroll
            for (int j = 0; j < HK; j += 2) {
                const float p0 = exp2f(s[j] - base), p1 = exp2f(s[j + 1] - base);
                l_run += p0 + p1;
                const __half2 h2 = __floats2half2_rn(p0, p1);
                const float2 hf = __half22float2(h2);
                const __half2 l2 = __floats2half2_rn(p0 - hf.x, p1 - hf.y);
                ph[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
                pl[j / 2] = *reinterpret_cast<const uint32_t*>(&l2);
            }
#pragma unroll
            for (int k8 = 0; k8 < HK / 8; ++k8) {
                const uint32_t off = tc::cm_offset(srow, half * HK + k8 * 8, kTK);
                *reinterpret_cast<uint4*>(Phi_s + off) = make_uint4(ph[4 * k8], ph[4 * k8 + 1], ph[4 * k8 + 2], ph[4 * k8 + 3]);
                *reinterpret_cast<uint4*>(Plo_s + off) = make_uint4(pl[4 * k8], pl[4 * k8 + 1], pl[4 * k8 + 2], pl[4 * k8 + 3]);
            }
            // O *= alpha for this row (tensor memory) when its max moved; the
            // two threads of a row take half of the columns each
            if (__any_sync(0xffffffffu, rescale) && ok) {
                const float al = rescale ? alpha : 1.f;
#pragma unroll 1
                for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
                    float o[32];
                    tc::ld32(tmem_O + lane_off + c0, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= al;
                    tc::st32(tmem_O + lane_off + c0, o);
                }
            }
            fence_proxy_async_smem();
        }
        tc::fence_before_sync();
        __syncthreads();

        // O += P_hi V_hi + P_hi V_lo + P_lo V_hi
        if (tid == 0 && !*fail_s) {
            tc::fence_after_sync();
            const uint32_t ph = smem_u32(Phi_s), pl = smem_u32(Plo_s), vh = smem_u32(Vhi_s), vl = smem_u32(Vlo_s);
            constexpr uint32_t P_SBO = (kTK / 8) * 128, V_LBO = (D / 8) * 128;
#pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks) {
                const uint64_t ah = tc::smem_desc(ph + ks * 256, 128, P_SBO);
                const uint64_t al = tc::smem_desc(pl + ks * 256, 128, P_SBO);
                const uint64_t bh = tc::smem_desc(vh + ks * 2 * V_LBO, V_LBO, 128);
                const uint64_t bl = tc::smem_desc(vl + ks * 2 * V_LBO, V_LBO, 128);
                tc::mma_f16(tmem_O, ah, bh, idesc_pv, o_valid || ks > 0);
                tc::mma_f16(tmem_O, ah, bl, idesc_pv, true);
                tc::mma_f16(tmem_O, al, bh, idesc_pv, true);
            }
            tc::commit(bar_o);
        }
        // every thread waits: the tile buffers and O are reused next
        if (!*fail_s && !wait_phase(bar_o, phase)) atomicOr(fail_s, 1);
        tc::fence_after_sync();
        o_valid = true;
        phase ^= 1;
    }
    cp_async_wait<0>();
    __syncthreads();
    if (*fail_s && tid == 0) raise_status(a.status, DFLV_DEV_TIMEOUT);

    // ---- partial results -> shared memory (reusing the tile region)
    float* Om = reinterpret_cast<float*>(smem + S::off_Om);
    float* Mm = reinterpret_cast<float*>(smem + S::off_Mm);
    float* Lm = reinterpret_cast<float*>(smem + S::off_Lm);
    xch_s[half * kRows + srow] = l_run;
    __syncthreads();
    {
#pragma unroll 1
        for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
            float o[32];
            if (o_valid && !*fail_s) tc::ld32(tmem_O + lane_off + c0, o);
            else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(Om + srow * OS + c0 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
        if (half == 0) {
            Mm[srow] = m_run;
            Lm[srow] = l_run + xch_s[kRows + srow];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, S::kTmemCols);
    cluster_sync_all();

    // ---- merge: rank r finalises rows r, r + CS, ... (one warp per row); a
    //      row's peer values are all requested before any is used
    const uint32_t om_base = smem_u32(Om), mm_base = smem_u32(Mm), lm_base = smem_u32(Lm);
    constexpr int nwarps = kThreads / 32;
    constexpr int PL = D / 32;  // output floats per lane
    for (int r = rank + CS * warp; r < RT; r += CS * nwarps) {
        const int rho = row0 + r;
        if (rho >= rows_valid) continue;
        float M = -INFINITY;
        for (int q = 0; q < CS; ++q) M = fmaxf(M, ld_dsmem_f32(map_to_rank(mm_base + r * 4, q)));
        const float bse = (M == -INFINITY) ? 0.f : M;
        float Lt = 0.f, acc[PL];
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] = 0.f;
        for (int q0 = 0; q0 < CS; q0 += 8) {  // peers in batches of eight
            float v[8][PL], mq[8], lq[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const bool on = q0 + q < CS;
                mq[q] = on ? ld_dsmem_f32(map_to_rank(mm_base + r * 4, q0 + q)) : -INFINITY;
                lq[q] = on ? ld_dsmem_f32(map_to_rank(lm_base + r * 4, q0 + q)) : 0.f;
#pragma unroll
                for (int e = 0; e < PL; e += 4) {
                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (on) x = ld_dsmem_f4(map_to_rank(om_base + (r * OS + lane * PL + e) * 4, q0 + q));
                    v[q][e] = x.x;
                    v[q][e + 1] = x.y;
                    v[q][e + 2] = x.z;
                    v[q][e + 3] = x.w;
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float w = exp2f(mq[q] - bse);  // 0 for absent peers (mq = -inf)
                Lt = fmaf(w, lq[q], Lt);
#pragma unroll
                for (int e = 0; e < PL; ++e) acc[e] = fmaf(w, v[q][e], acc[e]);
            }
        }
        const float inv = 1.f / Lt;
        const int i = rho / G, gh = rho % G;
        float* dst = a.out + (((size_t)b * N + i) * a.Hq + kvh * G + gh) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv, acc[e + 3] * inv);
    }
    cluster_sync_all();  // peers may still be reading this CTA's shared memory
}

// How many clusters of cs CTAs of this kernel can be resident at once at
// this shared-memory size (queried once per kernel and cluster size; 16 uses
// the non-portable cluster size).
template <typename Kernel>
int active_clusters(Kernel kern, size_t smem, int cs) {
    static int cache[17] = {0};
    if (cs < 1 || cs > 16) return 0;
    if (cache[cs] == 0) {
        int n = 0;
        if (cs > 8) cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
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

template <int D, int TYPE>
cudaError_t launch_tc(const AttnVerifyArgs& a, cudaStream_t stream) {
    using S = TcSmem<D, TYPE>;
    auto kern = attn_tc_kernel<D, TYPE>;
    cudaError_t e = ensure_smem(kern, S::total);
    if (e != cudaSuccess) return e;
    const int rows = (a.Hq / a.Hkv) * a.N_max;
    const int n_rt = (rows + kRows - 1) / kRows;
    const int RT = (rows + n_rt - 1) / n_rt;
    const long range = (a.window > 0) ? (long)a.window - 1 : (long)a.cap;
    const long tiles = (range + kTK - 1) / kTK + 2;
    const long clusters = (long)n_rt * a.Hkv * a.B;
    const int sms = sm_count_cached();
    // the largest cluster (<= 16) that still lets every cluster be resident
    // at once and that the key range can feed
    int cs = 1;
    while (cs < 16 && clusters * cs * 2 <= sms && cs * 2 <= tiles &&
           active_clusters(kern, S::total, cs * 2) >= clusters)
        cs *= 2;
    return launch_pdl(kern, dim3(cs, n_rt * a.Hkv, a.B), dim3(kThreads), S::total, stream, cs, a, RT, cs);
}

}  // namespace

cudaError_t launch_attn_tree_verify_tc(const AttnVerifyArgs& a, cudaStream_t stream) {
    const bool q8 = a.type == DFLV_KV_Q8_0;
    switch (a.D) {
        case 128: return q8 ? launch_tc<128, DFLV_KV_Q8_0>(a, stream) : launch_tc<128, DFLV_KV_Q4_0>(a, stream);
        case 256: return q8 ? launch_tc<256, DFLV_KV_Q8_0>(a, stream) : launch_tc<256, DFLV_KV_Q4_0>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dflv
