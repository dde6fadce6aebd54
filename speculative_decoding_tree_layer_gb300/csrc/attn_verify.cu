// attn_verify.cu -- tree verify of one full-attention layer over a
// block-quantised KV cache.
//
// What it computes (see include/dflv.h): the tree's keys/values are
// quantised into cache slots [P, P + n); then every (node i, query head h)
// attends, with softmax(q.k * scale), to the cached positions j < P inside
// its sliding window and to the tree slots of its ancestors-or-self ("Luce
// DFlash" README, "How it works": a causal mask derived from parent
// pointers; "--fa-window N", 0 = full attention; "Asymmetric K/V
// quantization": q8_0 default, Q4_0).  Node i sits at position
// P + depth(i); a key at position j is visible iff j <= that position and
// (W == 0 or j > position - W).
//
// How (q8_0 / q4_0):
//   * quantise kernel: one warp per (sequence, node, KV head) writes the
//     node's K and V rows into their slots (fp32 amax, IEEE division, fp16
//     scale, round-half-away codes), so the tree attends exactly what a
//     sequential decode would have stored;
//   * main kernel: one thread-block CLUSTER per (sequence, KV head, row
//     tile).  A row tile holds up to 128 query rows (every query head of the
//     group x every node), so each KV byte is read once per row tile.  The
//     cluster's CTAs split the visible key range [lo, P) plus the tree block
//     into 64-key tiles (split-K), stream them through shared memory with
//     16-byte cp.async double buffering, and run q.k on the tensor cores:
//     int8 / 4-bit codes become fp16 exactly in registers and the per-block
//     fp16 scale is applied to the fp32 accumulator of each 32-dim block, so
//     the scores are exact up to fp32 accumulation.  V codes are staged in
//     shared memory as exact fp16 integers and each key's block scale is
//     folded into its softmax weight (p * d_v, rounded once to fp16) right
//     before p.V runs on the tensor cores, with an fp32 online softmax.
//     Rounding dequantised V to fp16 instead would add a second rounding
//     per term and roughly triple the worst-case output error.  The per-CTA partial (max, sum,
//     output) are merged through distributed shared memory -- no global
//     scratch and no second launch.
// f32 caches (small exactness checks) take a plain CUDA-core kernel.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tree.cuh"

namespace dflv {

namespace {

constexpr int kTileKeys = 64;
constexpr int kMaxRowTile = 128;  // 8 warps x 16 rows (two warps per SM sub-partition keep 255 registers)
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- cluster helpers
DFLV_DEVINL uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
DFLV_DEVINL void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                     : "memory");
}
DFLV_DEVINL uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
DFLV_DEVINL float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
DFLV_DEVINL float2 ld_dsmem_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0,%1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// ---------------------------------------------------------------- exact code -> fp16
// fp16 with exponent field 25 (0x6400 = 1024) has unit spacing on
// [1024, 2048): the bit pattern 0x6400 | u is exactly 1024 + u for u < 1024.
DFLV_DEVINL uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// four int8 codes -> {c0,c1}, {c2,c3} as exact fp16x2
DFLV_DEVINL void i8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;  // code + 128 in [1, 255]
    const uint32_t l = prmt(u, 0x64646464u, 0x5140u);
    const uint32_t h = prmt(u, 0x64646464u, 0x5342u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 lh = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
    __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
    lo = *reinterpret_cast<uint32_t*>(&lh);
    hi = *reinterpret_cast<uint32_t*>(&hh);
}
// four 4-bit codes (one per byte, low nibble) -> value - 8 as exact fp16x2
DFLV_DEVINL void u4x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t l = prmt(w, 0x64646464u, 0x5140u);
    const uint32_t h = prmt(w, 0x64646464u, 0x5342u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
    __half2 lh = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
    __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
    lo = *reinterpret_cast<uint32_t*>(&lh);
    hi = *reinterpret_cast<uint32_t*>(&hh);
}

// ---------------------------------------------------------------- quantise tree K/V into the cache
// q8_0: d = fp16(amax / 127), code = clamp(round_half_away(x / d), -127, 127)
// q4_0: d = fp16(amax / 7),   code = clamp(round_half_away(x / d), -8, 7) + 8,
//       element j < 16 in the low nibble of byte j, element j + 16 in its high nibble.
__global__ void attn_quantize_tree_kernel(AttnVerifyArgs a) {
    const int i = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    grid_dependency_wait();
    const int n = __ldg(a.n_nodes + b), P = __ldg(a.n_past + b);
    if (n < 1 || n > a.N_max) return;  // reported by the attention kernel
    if (P < 0 || P + n > a.cap) return;
    if (i >= n) return;
    const size_t src_row = (((size_t)b * a.N_max + i) * a.Hkv + kvh) * a.D;
    const size_t dst_row = ((size_t)b * a.Hkv + kvh) * a.cap + P + i;
    if (a.type == DFLV_KV_F32) {
        for (int t = threadIdx.x; t < 2 * a.D; t += blockDim.x) {
            const int which = t / a.D, d = t % a.D;
            const uint16_t* src = which ? a.v_new : a.k_new;
            float* dst = reinterpret_cast<float*>(which ? a.vq : a.kq);
            dst[dst_row * a.D + d] = bf16_bits_to_float(src[src_row + d]);
        }
        return;
    }
    const int nb = a.D / 32;
    const bool q8 = a.type == DFLV_KV_Q8_0;
    for (int t = threadIdx.x; t < 2 * nb; t += blockDim.x) {
        const int which = t / nb, blk = t % nb;
        const uint16_t* src = (which ? a.v_new : a.k_new) + src_row + blk * 32;
        float x[32];
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            x[j] = bf16_bits_to_float(src[j]);
            amax = fmaxf(amax, fabsf(x[j]));
        }
        const float d = __fdiv_rn(amax, q8 ? 127.f : 7.f);
        const __half dh = __float2half_rn(d);
        const float df = __half2float(dh);
        uint16_t* sc = which ? a.vs : a.ks;
        sc[dst_row * nb + blk] = __half_as_ushort(dh);
        uint8_t* plane = reinterpret_cast<uint8_t*>(which ? a.vq : a.kq);
        if (q8) {
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float r = (df == 0.f) ? 0.f : roundf(__fdiv_rn(x[j], df));
                r = fminf(fmaxf(r, -127.f), 127.f);
                const uint32_t c = (uint32_t)(uint8_t)(int8_t)(int)r;
                if ((j & 3) == 0) w[j >> 2] = 0;
                w[j >> 2] |= c << (8 * (j & 3));
            }
            uint4* dst = reinterpret_cast<uint4*>(plane + dst_row * a.D + blk * 32);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
            uint32_t code[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float r = (df == 0.f) ? 0.f : roundf(__fdiv_rn(x[j], df));
                r = fminf(fmaxf(r, -8.f), 7.f);
                code[j] = (uint32_t)((int)r + 8);
            }
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t byte = code[j] | (code[j + 16] << 4);
                if ((j & 3) == 0) w[j >> 2] = 0;
                w[j >> 2] |= byte << (8 * (j & 3));
            }
            *reinterpret_cast<uint4*>(plane + dst_row * (a.D / 2) + blk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// ---------------------------------------------------------------- main kernel (q8_0 / q4_0)
template <int D, int TYPE>
struct AttnSmem {
    static constexpr int NB = D / 32;                                  // scale blocks per row
    static constexpr int KB = (TYPE == DFLV_KV_Q8_0) ? D : D / 2;      // code bytes per row
    static constexpr int KSB = KB + 16;                                // padded K row (bytes)
    static constexpr int QS = D + 16;                                  // Q row stride (halves)
    static constexpr int VS = D + 8;                                   // dequantised V row stride (halves)
    static constexpr int OS = D + 4;                                   // merge row stride (floats)
    static constexpr size_t kHeader = 2048;
    // per-buffer tile bytes
    static constexpr size_t kK = (size_t)kTileKeys * KSB;
    static constexpr size_t kKs = (size_t)kTileKeys * NB * 2;
    static constexpr size_t kV = (size_t)kTileKeys * KB;
    static constexpr size_t kVs = (size_t)kTileKeys * NB * 2;
    static size_t __host__ __device__ off_Q() { return kHeader; }
    static size_t __host__ __device__ off_K(int RT) { return kHeader + (size_t)RT * QS * 2; }
    static size_t __host__ __device__ off_Ks(int RT) { return off_K(RT) + 2 * kK; }
    static size_t __host__ __device__ off_V(int RT) { return off_Ks(RT) + 2 * kKs; }
    static size_t __host__ __device__ off_Vs(int RT) { return off_V(RT) + 2 * kV; }
    static size_t __host__ __device__ off_Vh(int RT) { return off_Vs(RT) + 2 * kVs; }
    static size_t __host__ __device__ off_VsT(int RT) { return off_Vh(RT) + (size_t)kTileKeys * VS * 2; }
    static size_t __host__ __device__ loop_total(int RT) { return off_VsT(RT) + (size_t)NB * kTileKeys * 4; }
    // merge buffers reuse the region from off_Q once the tile loop is done
    static size_t __host__ __device__ off_Om() { return kHeader; }
    static size_t __host__ __device__ off_Mm(int RT) { return kHeader + (size_t)RT * OS * 4; }
    static size_t __host__ __device__ off_Lm(int RT) { return off_Mm(RT) + (size_t)RT * 4; }
    static size_t __host__ __device__ merge_total(int RT) { return off_Lm(RT) + (size_t)RT * 4; }
    static size_t __host__ __device__ total(int RT) {
        size_t a = loop_total(RT), b = merge_total(RT);
        return a > b ? a : b;
    }
};

template <int D, int TYPE>
__global__ void __launch_bounds__(kMaxRowTile * 2, 1)
    attn_tree_verify_kernel(AttnVerifyArgs a, int RT, int CS) {
    using S = AttnSmem<D, TYPE>;
    constexpr int NB = S::NB, KB = S::KB, KSB = S::KSB, QS = S::QS, VS = S::VS, OS = S::OS;
    extern __shared__ __align__(128) unsigned char smem[];
    int32_t* par_s = reinterpret_cast<int32_t*>(smem);
    int32_t* depth_s = par_s + kMaxNodes;
    uint64_t* amask_s = reinterpret_cast<uint64_t*>(smem + 512);
    uint16_t* Q_s = reinterpret_cast<uint16_t*>(smem + S::off_Q());
    uint8_t* K_s = smem + S::off_K(RT);
    uint16_t* Ks_s = reinterpret_cast<uint16_t*>(smem + S::off_Ks(RT));
    uint8_t* V_s = smem + S::off_V(RT);
    uint16_t* Vs_s = reinterpret_cast<uint16_t*>(smem + S::off_Vs(RT));
    uint16_t* Vh_s = reinterpret_cast<uint16_t*>(smem + S::off_Vh(RT));
    float* VsT_s = reinterpret_cast<float*>(smem + S::off_VsT(RT));  // [NB][64] V block scales

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int gq = lane >> 2, tq = lane & 3;
    const int rank = (int)cluster_ctarank();
    const int kvh = blockIdx.y % a.Hkv, rt = blockIdx.y / a.Hkv, b = blockIdx.z;
    const int G = a.Hq / a.Hkv, N = a.N_max, W = a.window;

    grid_dependency_wait();
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
        return;

    const size_t plane_row0 = ((size_t)b * a.Hkv + kvh) * a.cap;  // slot 0 of this (seq, kv head)
    const uint8_t* kq = reinterpret_cast<const uint8_t*>(a.kq);
    const uint8_t* vq = reinterpret_cast<const uint8_t*>(a.vq);

    // Tiles: cache keys [lo, P) in 64-key tiles, then one tree tile [P, P + n).
    const int lo = (W > 0) ? max(0, P - W + 1) : 0;
    const int n_cache_tiles = (P - lo + kTileKeys - 1) / kTileKeys;
    const int n_tiles = n_cache_tiles + 1;

    auto issue_tile = [&](int t, int buf) {
        const int start = (t < n_cache_tiles) ? lo + t * kTileKeys : P;
        const int count = (t < n_cache_tiles) ? min(kTileKeys, P - start) : n;
        uint8_t* kd = K_s + buf * S::kK;
        uint8_t* vd = V_s + buf * S::kV;
        uint8_t* ksd = reinterpret_cast<uint8_t*>(Ks_s) + buf * S::kKs;
        uint8_t* vsd = reinterpret_cast<uint8_t*>(Vs_s) + buf * S::kVs;
        constexpr int CPR = KB / 16;  // 16-byte chunks per code row
        for (int idx = tid; idx < count * CPR; idx += nthreads) {
            const int c = idx / CPR, ch = idx % CPR;
            const size_t g = (plane_row0 + start + c) * KB + ch * 16;
            cp_async16(kd + c * KSB + ch * 16, kq + g);
            cp_async16(vd + c * KB + ch * 16, vq + g);
        }
        // scale rows: NB halves = 2*NB bytes each (4, 8 or 16: one cp.async per row)
        for (int c = tid; c < count; c += nthreads) {
            const size_t g = (plane_row0 + start + c) * NB;
            if constexpr (NB * 2 == 16) {
                cp_async16(ksd + c * 16, a.ks + g);
                cp_async16(vsd + c * 16, a.vs + g);
            } else if constexpr (NB * 2 == 8) {
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(ksd + c * 8)), "l"(a.ks + g) : "memory");
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(vsd + c * 8)), "l"(a.vs + g) : "memory");
            } else {
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(ksd + c * 4)), "l"(a.ks + g) : "memory");
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(vsd + c * 4)), "l"(a.vs + g) : "memory");
            }
        }
        cp_async_commit();
    };

    // First tile of this CTA in flight before the query rows load.
    int t_cur = rank;
    if (t_cur < n_tiles) issue_tile(t_cur, 0);
    else cp_async_commit();

    // Query rows of this tile: row r <-> flat (node i, head gh) = row0 + r = i * G + gh.
    const int nwarps = nthreads / 32;
    const int RTw = nwarps * 16;  // rows covered by the warps (== RT)
    for (int idx = tid; idx < RTw * (D / 8); idx += nthreads) {
        const int r = idx / (D / 8), c8 = idx % (D / 8);
        const int rho = row0 + r;
        uint4 outv = make_uint4(0, 0, 0, 0);
        if (rho < rows_valid) {
            const int i = rho / G, gh = rho % G;
            const uint4 inv = __ldg(reinterpret_cast<const uint4*>(
                a.q + (((size_t)b * N + i) * a.Hq + kvh * G + gh) * D + c8 * 8));
            const uint32_t w[4] = {inv.x, inv.y, inv.z, inv.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = pack_f16x2(bf16_bits_to_float((uint16_t)(w[e] & 0xffff)),
                                  bf16_bits_to_float((uint16_t)(w[e] >> 16)));
            outv = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(Q_s + r * QS + c8 * 8) = outv;
    }

    // Per-thread row metadata: rows gq and gq + 8 of this warp.
    int rnode[2], lb[2], rdepth[2];
    uint64_t ramask[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int rho = row0 + warp * 16 + gq + 8 * s;
        if (rho < rows_valid) {
            const int i = rho / G;
            rnode[s] = i;
            rdepth[s] = depth_s[i];
            ramask[s] = amask_s[i];
            lb[s] = (W > 0) ? P + depth_s[i] - W + 1 : INT_MIN;
        } else {
            rnode[s] = -1;
            rdepth[s] = 0;
            ramask[s] = 0;
            lb[s] = INT_MAX;
        }
    }

    const float sl2 = a.scale * kLog2e;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float O[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) O[j][0] = O[j][1] = O[j][2] = O[j][3] = 0.f;

    int buf = 0;
    for (; t_cur < n_tiles; t_cur += CS, buf ^= 1) {
        const int t_next = t_cur + CS;
        if (t_next < n_tiles) issue_tile(t_next, buf ^ 1);
        else cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const bool tree_tile = t_cur >= n_cache_tiles;
        const int start = tree_tile ? P : lo + t_cur * kTileKeys;
        const int count = tree_tile ? n : min(kTileKeys, P - start);
        const uint8_t* kb = K_s + buf * S::kK;
        const uint16_t* ksb = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(Ks_s) + buf * S::kKs);
        const uint8_t* vb = V_s + buf * S::kV;
        const uint16_t* vsb = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(Vs_s) + buf * S::kVs);

        // V codes -> exact fp16 integers (rows past count are zero); block
        // scales transposed to [block][key] in fp32 (zero past count)
        for (int idx = tid; idx < kTileKeys * (D / 8); idx += nthreads) {
            const int c = idx / (D / 8), d8 = idx % (D / 8);
            uint4 o = make_uint4(0, 0, 0, 0);
            if (c < count) {
                if constexpr (TYPE == DFLV_KV_Q8_0) {
                    const uint2 w = *reinterpret_cast<const uint2*>(vb + c * KB + d8 * 8);
                    i8x4_to_f16x2(w.x, o.x, o.y);
                    i8x4_to_f16x2(w.y, o.z, o.w);
                } else {
                    // dims d8*8 .. d8*8+7 of 32-block blk sit in the low (first
                    // half of the block) or high nibbles of 8 consecutive bytes
                    const int blk = (d8 * 8) / 32, off = (d8 * 8) % 32;
                    const uint2 w = *reinterpret_cast<const uint2*>(vb + c * KB + blk * 16 + (off & 15));
                    const int sh = off >= 16 ? 4 : 0;
                    u4x4_to_f16x2((w.x >> sh) & 0x0f0f0f0fu, o.x, o.y);
                    u4x4_to_f16x2((w.y >> sh) & 0x0f0f0f0fu, o.z, o.w);
                }
            }
            *reinterpret_cast<uint4*>(Vh_s + c * VS + d8 * 8) = o;
        }
        for (int idx = tid; idx < NB * kTileKeys; idx += nthreads) {
            const int blk = idx / kTileKeys, c = idx % kTileKeys;
            VsT_s[idx] = (c < count) ? __half2float(__ushort_as_half(vsb[c * NB + blk])) : 0.f;
        }

        // scores: S = sum over 32-dim blocks of scale_k * (q . codes), on tensor cores
        float Sacc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) Sacc[nt][0] = Sacc[nt][1] = Sacc[nt][2] = Sacc[nt][3] = 0.f;
        const uint16_t* q0 = Q_s + (warp * 16 + gq) * QS;
        const uint16_t* q1 = q0 + 8 * QS;
#pragma unroll 1
        for (int blk = 0; blk < NB; ++blk) {
            uint32_t qa[2][4];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int col = (2 * blk + kk) * 16 + tq * 4;
                const uint2 r0 = *reinterpret_cast<const uint2*>(q0 + col);
                const uint2 r1 = *reinterpret_cast<const uint2*>(q1 + col);
                qa[kk][0] = r0.x;
                qa[kk][1] = r1.x;
                qa[kk][2] = r0.y;
                qa[kk][3] = r1.y;
            }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const uint8_t* krow = kb + (nt * 8 + gq) * KSB;
                uint32_t bfr[2][2];
                if constexpr (TYPE == DFLV_KV_Q8_0) {
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(krow + (2 * blk) * 16 + tq * 4);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(krow + (2 * blk + 1) * 16 + tq * 4);
                    i8x4_to_f16x2(w0, bfr[0][0], bfr[0][1]);
                    i8x4_to_f16x2(w1, bfr[1][0], bfr[1][1]);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(krow + blk * 16 + tq * 4);
                    u4x4_to_f16x2(w & 0x0f0f0f0fu, bfr[0][0], bfr[0][1]);
                    u4x4_to_f16x2((w >> 4) & 0x0f0f0f0fu, bfr[1][0], bfr[1][1]);
                }
                float t4[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16_16816(t4, qa[0], bfr[0]);
                mma_f16_16816(t4, qa[1], bfr[1]);
                const int key = nt * 8 + tq * 2;
                const float s0 = __half2float(__ushort_as_half(ksb[key * NB + blk]));
                const float s1 = __half2float(__ushort_as_half(ksb[(key + 1) * NB + blk]));
                Sacc[nt][0] = fmaf(t4[0], s0, Sacc[nt][0]);
                Sacc[nt][1] = fmaf(t4[1], s1, Sacc[nt][1]);
                Sacc[nt][2] = fmaf(t4[2], s0, Sacc[nt][2]);
                Sacc[nt][3] = fmaf(t4[3], s1, Sacc[nt][3]);
            }
        }

        // mask + online softmax (log2 domain)
        float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int s = c >> 1;
                const int key = nt * 8 + tq * 2 + (c & 1);
                bool vis;
                if (tree_tile) {
                    vis = key < count && ((ramask[s] >> key) & 1ull) &&
                          (W == 0 || depth_s[key] > rdepth[s] - W);
                } else {
                    vis = key < count && start + key >= lb[s];
                }
                const float v = vis ? Sacc[nt][c] * sl2 : -INFINITY;
                Sacc[nt][c] = v;
                mt[s] = fmaxf(mt[s], v);
            }
        float alpha[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            mt[s] = fmaxf(mt[s], __shfl_xor_sync(0xffffffffu, mt[s], 1));
            mt[s] = fmaxf(mt[s], __shfl_xor_sync(0xffffffffu, mt[s], 2));
            const float m_new = fmaxf(m_run[s], mt[s]);
            const float base = (m_new == -INFINITY) ? 0.f : m_new;
            alpha[s] = exp2f(m_run[s] - base);
            m_run[s] = m_new;
            mt[s] = base;
            l_run[s] *= alpha[s];
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int s = c >> 1;
                const float p = exp2f(Sacc[nt][c] - mt[s]);
                Sacc[nt][c] = p;
                l_run[s] += p;
            }
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            O[j][0] *= alpha[0];
            O[j][1] *= alpha[0];
            O[j][2] *= alpha[1];
            O[j][3] *= alpha[1];
        }
        __syncthreads();  // V codes and scales staged

        // O += (P * d_v) V_codes on tensor cores, one 32-dim V block at a time
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const uint32_t base = smem_u32(Vh_s + key * VS + (lane >> 4) * 8);
            const int k01 = kk * 16 + tq * 2;
#pragma unroll
            for (int blk = 0; blk < NB; ++blk) {
                const float2 s01 = *reinterpret_cast<const float2*>(VsT_s + blk * kTileKeys + k01);
                const float2 s89 = *reinterpret_cast<const float2*>(VsT_s + blk * kTileKeys + k01 + 8);
                uint32_t pa[4];
                pa[0] = pack_f16x2(Sacc[2 * kk][0] * s01.x, Sacc[2 * kk][1] * s01.y);
                pa[1] = pack_f16x2(Sacc[2 * kk][2] * s01.x, Sacc[2 * kk][3] * s01.y);
                pa[2] = pack_f16x2(Sacc[2 * kk + 1][0] * s89.x, Sacc[2 * kk + 1][1] * s89.y);
                pa[3] = pack_f16x2(Sacc[2 * kk + 1][2] * s89.x, Sacc[2 * kk + 1][3] * s89.y);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int dn = 2 * blk + half;
                    uint32_t r[4];
                    ldmatrix_x4_trans(r, base + dn * 16 * 2);
                    const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
                    mma_f16_16816(O[2 * dn], pa, b0);
                    mma_f16_16816(O[2 * dn + 1], pa, b1);
                }
            }
        }
        __syncthreads();  // buffers free for the next prefetch
    }
    cp_async_wait<0>();

    // per-row partial results -> shared memory (reusing the tile region)
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        l_run[s] += __shfl_xor_sync(0xffffffffu, l_run[s], 1);
        l_run[s] += __shfl_xor_sync(0xffffffffu, l_run[s], 2);
    }
    __syncthreads();
    float* Om = reinterpret_cast<float*>(smem + S::off_Om());
    float* Mm = reinterpret_cast<float*>(smem + S::off_Mm(RT));
    float* Lm = reinterpret_cast<float*>(smem + S::off_Lm(RT));
    {
        const int r0 = warp * 16 + gq;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            *reinterpret_cast<float2*>(Om + r0 * OS + j * 8 + tq * 2) = make_float2(O[j][0], O[j][1]);
            *reinterpret_cast<float2*>(Om + (r0 + 8) * OS + j * 8 + tq * 2) = make_float2(O[j][2], O[j][3]);
        }
        if (tq == 0) {
            Mm[r0] = m_run[0];
            Mm[r0 + 8] = m_run[1];
            Lm[r0] = l_run[0];
            Lm[r0 + 8] = l_run[1];
        }
    }
    cluster_sync_all();

    // merge: rank r finalises rows r, r + CS, ... (one warp per row)
    const uint32_t om_base = smem_u32(Om), mm_base = smem_u32(Mm), lm_base = smem_u32(Lm);
    for (int r = rank + CS * warp; r < RTw; r += CS * nwarps) {
        const int rho = row0 + r;
        if (rho >= rows_valid) continue;
        float M = -INFINITY;
        for (int q = 0; q < CS; ++q) M = fmaxf(M, ld_dsmem_f32(map_to_rank(mm_base + r * 4, q)));
        const float base = (M == -INFINITY) ? 0.f : M;
        float Lt = 0.f;
        constexpr int PL = D / 32;  // output floats per lane (2, 4 or 8), as PL/2 float2
        float2 acc[PL / 2];
#pragma unroll
        for (int e = 0; e < PL / 2; ++e) acc[e] = make_float2(0.f, 0.f);
        for (int q = 0; q < CS; ++q) {
            const float w = exp2f(ld_dsmem_f32(map_to_rank(mm_base + r * 4, q)) - base);
            Lt = fmaf(w, ld_dsmem_f32(map_to_rank(lm_base + r * 4, q)), Lt);
#pragma unroll
            for (int e = 0; e < PL / 2; ++e) {
                const float2 v = ld_dsmem_f2(map_to_rank(om_base + (r * OS + lane * PL + 2 * e) * 4, q));
                acc[e].x = fmaf(w, v.x, acc[e].x);
                acc[e].y = fmaf(w, v.y, acc[e].y);
            }
        }
        const float inv = 1.f / Lt;
        const int i = rho / G, gh = rho % G;
        float* dst = a.out + (((size_t)b * N + i) * a.Hq + kvh * G + gh) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL / 2; ++e)
            *reinterpret_cast<float2*>(dst + 2 * e) = make_float2(acc[e].x * inv, acc[e].y * inv);
    }
    cluster_sync_all();  // peers may still be reading this CTA's shared memory
}

// ---------------------------------------------------------------- f32 cache (CUDA cores)
// One warp per (sequence, node, query head); keys in chunks of 32 (one per
// lane), online softmax across the warp, output dims strided over lanes.
__global__ void attn_tree_verify_f32_kernel(AttnVerifyArgs a) {
    __shared__ int32_t par_s[kMaxNodes], depth_s[kMaxNodes];
    __shared__ uint64_t amask_s[kMaxNodes];
    __shared__ float q_s[8][256];
    const int b = blockIdx.z, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + warp;
    const int N = a.N_max, D = a.D, W = a.window, G = a.Hq / a.Hkv, kvh = h / G;
    grid_dependency_wait();
    const int n = __ldg(a.n_nodes + b), P = __ldg(a.n_past + b);
    if (P < 0 || P + n > a.cap || n < 1 || n > N) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0)
            raise_status(a.status, (n < 1 || n > N) ? DFLV_DEV_TOPOLOGY : DFLV_DEV_CAPACITY);
        return;
    }
    if (!block_tree_topology(a.parent + (size_t)b * N, n, N, par_s, depth_s, amask_s,
                             (blockIdx.x == 0 && h == 0) ? a.status : nullptr))
        return;
    if (i >= n) return;
    for (int d = lane; d < D; d += 32)
        q_s[warp][d] = bf16_bits_to_float(a.q[(((size_t)b * N + i) * a.Hq + h) * D + d]);
    __syncwarp();
    const float* K = reinterpret_cast<const float*>(a.kq) + ((size_t)b * a.Hkv + kvh) * a.cap * D;
    const float* V = reinterpret_cast<const float*>(a.vq) + ((size_t)b * a.Hkv + kvh) * a.cap * D;
    const int ipos = P + depth_s[i];
    const uint64_t am = amask_s[i];
    float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int base = 0; base < P + n; base += 32) {
        const int slot = base + lane;
        bool vis = false;
        if (slot < P) {
            vis = (W == 0) || slot > ipos - W;
        } else if (slot < P + n) {
            const int l_ = slot - P;
            vis = ((am >> l_) & 1ull) && ((W == 0) || P + depth_s[l_] > ipos - W);
        }
        float s = -INFINITY;
        if (vis) {
            float dot = 0.f;
            for (int d = 0; d < D; ++d) dot = fmaf(q_s[warp][d], K[(size_t)slot * D + d], dot);
            s = dot * a.scale;
        }
        float cm = s;
        for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        const float m_new = fmaxf(m, cm);
        const float base_m = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = expf(m - base_m);
        const float p = expf(s - base_m);
        float ps = p;
        for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l = l * alpha + ps;
        m = m_new;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= alpha;
        for (int j = 0; j < 32; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, j);
            if (pj == 0.f) continue;
            const int sj = base + j;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int d = lane + 32 * e;
                if (d < D) acc[e] = fmaf(pj, V[(size_t)sj * D + d], acc[e]);
            }
        }
    }
    float* dst = a.out + (((size_t)b * N + i) * a.Hq + h) * D;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int d = lane + 32 * e;
        if (d < D) dst[d] = acc[e] / l;
    }
}

// ---------------------------------------------------------------- launch
struct RowTiling {
    int RT, n_rt, CS;
};

RowTiling choose_tiling(const AttnVerifyArgs& a, int sm_count) {
    const int G = a.Hq / a.Hkv;
    const int rows = G * a.N_max;
    RowTiling t;
    t.n_rt = (rows + kMaxRowTile - 1) / kMaxRowTile;
    const int per = (rows + t.n_rt - 1) / t.n_rt;
    t.RT = ((per + 15) / 16) * 16;
    const long range = (a.window > 0) ? (long)a.window - 1 : (long)a.cap;
    const long tiles = (range + kTileKeys - 1) / kTileKeys + 1;
    const long clusters = (long)t.n_rt * a.Hkv * a.B;
    int cs = 1;
    while (cs < 8 && clusters * cs * 2 <= sm_count && cs * 2 <= tiles) cs *= 2;
    t.CS = cs;
    return t;
}

template <int D, int TYPE>
cudaError_t launch_main(const AttnVerifyArgs& a, cudaStream_t stream) {
    using S = AttnSmem<D, TYPE>;
    const RowTiling t = choose_tiling(a, sm_count_cached());
    const size_t smem = S::total(t.RT);
    auto kern = attn_tree_verify_kernel<D, TYPE>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(t.CS, t.n_rt * a.Hkv, a.B);
    cfg.blockDim = dim3(t.RT * 2, 1, 1);  // RT / 16 warps
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = t.CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, t.RT, t.CS);
}

}  // namespace

size_t attn_verify_smem_bytes(int D, int type, int RT) {
    if (type == DFLV_KV_Q8_0) {
        if (D == 64) return AttnSmem<64, DFLV_KV_Q8_0>::total(RT);
        if (D == 128) return AttnSmem<128, DFLV_KV_Q8_0>::total(RT);
        return AttnSmem<256, DFLV_KV_Q8_0>::total(RT);
    }
    if (D == 64) return AttnSmem<64, DFLV_KV_Q4_0>::total(RT);
    if (D == 128) return AttnSmem<128, DFLV_KV_Q4_0>::total(RT);
    return AttnSmem<256, DFLV_KV_Q4_0>::total(RT);
}

cudaError_t launch_attn_tree_verify(const AttnVerifyArgs& a, cudaStream_t stream) {
    attn_quantize_tree_kernel<<<dim3(a.N_max, a.Hkv, a.B), 32, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.type == DFLV_KV_F32) {
        attn_tree_verify_f32_kernel<<<dim3((a.N_max + 7) / 8, a.Hq, a.B), 256, 0, stream>>>(a);
        return cudaGetLastError();
    }
    const bool q8 = a.type == DFLV_KV_Q8_0;
    switch (a.D) {
        case 64: return q8 ? launch_main<64, DFLV_KV_Q8_0>(a, stream) : launch_main<64, DFLV_KV_Q4_0>(a, stream);
        case 128: return q8 ? launch_main<128, DFLV_KV_Q8_0>(a, stream) : launch_main<128, DFLV_KV_Q4_0>(a, stream);
        case 256: return q8 ? launch_main<256, DFLV_KV_Q8_0>(a, stream) : launch_main<256, DFLV_KV_Q4_0>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dflv
