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
// How (q8_0 / q4_0): one thread-block CLUSTER per (sequence, KV head, row
// tile).  A row tile holds up to 128 query rows (query heads of the group x
// nodes), so each KV byte is read once per row tile.
//   * Every CTA of the cluster first quantises its share of the tree's rows
//     into cache slots [P, P + n) (q8_0: d = amax / 127, q4_0: d = amax / 7,
//     stored as fp16; codes = round-half-away(x * (1/d)) from the fp32 d),
//     then the cluster synchronises, so the tree attends exactly what a
//     sequential decode would have stored and no extra launch is needed.
//   * The cluster's CTAs split the visible key range [lo, P) plus the tree
//     block into 64-key tiles (split-K) and stream them through shared
//     memory with 16-byte cp.async double buffering.  Each tile's int8 /
//     4-bit codes are staged once as exact fp16 integers (shared by all
//     warps) with the block scales transposed to fp32.
//   * q . k runs on the tensor cores (operands via ldmatrix) one 32-dim
//     block at a time, and each block's fp32 partial is scaled by the key's
//     block scale, so the scores are exact up to fp32 accumulation.
//   * fp32 online softmax; each key's V block scale is folded into its
//     softmax weight (p * d_v, rounded once to fp16) right before p . V on
//     the tensor cores.  (Rounding dequantised V to fp16 instead adds a
//     second rounding per term and roughly triples the worst-case error.)
//   * The per-CTA partial (max, sum, output) are merged through distributed
//     shared memory -- no global scratch.
// f32 caches (small exactness checks) take a plain CUDA-core kernel after a
// tiny kernel copies the tree's rows into the cache.
#include <climits>

#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tree.cuh"

namespace dflv {

namespace {

constexpr int kTileKeys = 64;
constexpr int kMaxRowTile = 128;  // 8 warps x 16 rows (two warps per SM sub-partition keep 255 registers)

using namespace attn;

// ---------------------------------------------------------------- f32 tree rows into the cache
__global__ void attn_store_tree_f32_kernel(AttnVerifyArgs a) {
    const int i = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    grid_dependency_wait();
    grid_launch_dependents();
    const int n = __ldg(a.n_nodes + b), P = __ldg(a.n_past + b);
    if (n < 1 || n > a.N_max || P < 0 || P + n > a.cap || i >= n) return;  // reported by the attention kernel
    const size_t src_row = (((size_t)b * a.N_max + i) * a.Hkv + kvh) * a.D;
    const size_t dst_row = ((size_t)b * a.Hkv + kvh) * a.cap + P + i;
    for (int t = threadIdx.x; t < 2 * a.D; t += blockDim.x) {
        const int which = t / a.D, d = t % a.D;
        const uint16_t* src = which ? a.v_new : a.k_new;
        float* dst = reinterpret_cast<float*>(which ? a.vq : a.kq);
        dst[dst_row * a.D + d] = bf16_bits_to_float(src[src_row + d]);
    }
}

// ---------------------------------------------------------------- main kernel (q8_0 / q4_0)
template <int D, int TYPE>
struct AttnSmem {
    static constexpr int NB = D / 32;                                  // scale blocks per row
    static constexpr int KB = (TYPE == DFLV_KV_Q8_0) ? D : D / 2;      // code bytes per row
    static constexpr int HS = D + 8;                                   // fp16 row stride (halves): conflict-free ldmatrix
    static constexpr int OS = D + 4;                                   // merge row stride (floats)
    static constexpr size_t kHeader = 2048;
    static constexpr size_t kRawCodes = (size_t)kTileKeys * KB;        // one plane of one tile
    static constexpr size_t kRawScales = (size_t)kTileKeys * NB * 2;
    static constexpr size_t kRawTile = 2 * kRawCodes + 2 * kRawScales; // K and V, codes and scales
    static size_t __host__ __device__ off_Q() { return kHeader; }
    static size_t __host__ __device__ off_raw(int RT) { return kHeader + (size_t)RT * HS * 2; }
    static size_t __host__ __device__ off_Kh(int RT) { return off_raw(RT) + 2 * kRawTile; }
    static size_t __host__ __device__ off_Vh(int RT) { return off_Kh(RT) + (size_t)kTileKeys * HS * 2; }
    static size_t __host__ __device__ off_KsT(int RT) { return off_Vh(RT) + (size_t)kTileKeys * HS * 2; }
    static size_t __host__ __device__ off_VsT(int RT) { return off_KsT(RT) + (size_t)NB * kTileKeys * 4; }
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
    constexpr int NB = S::NB, KB = S::KB, HS = S::HS, OS = S::OS;
    extern __shared__ __align__(128) unsigned char smem[];
    int32_t* par_s = reinterpret_cast<int32_t*>(smem);
    int32_t* depth_s = par_s + kMaxNodes;
    uint64_t* amask_s = reinterpret_cast<uint64_t*>(smem + 512);
    uint16_t* Q_s = reinterpret_cast<uint16_t*>(smem + S::off_Q());
    uint8_t* raw_s = smem + S::off_raw(RT);
    uint16_t* Kh_s = reinterpret_cast<uint16_t*>(smem + S::off_Kh(RT));
    uint16_t* Vh_s = reinterpret_cast<uint16_t*>(smem + S::off_Vh(RT));
    float* KsT_s = reinterpret_cast<float*>(smem + S::off_KsT(RT));  // [NB][64] K block scales
    float* VsT_s = reinterpret_cast<float*>(smem + S::off_VsT(RT));  // [NB][64] V block scales

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int gq = lane >> 2, tq = lane & 3;
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

    const size_t plane_row0 = ((size_t)b * a.Hkv + kvh) * a.cap;  // slot 0 of this (seq, kv head)
    uint8_t* kq = reinterpret_cast<uint8_t*>(a.kq);
    uint8_t* vq = reinterpret_cast<uint8_t*>(a.vq);

    // Tiles: cache keys [lo, P) in 64-key tiles, then one tree tile [P, P + n).
    const int lo = (W > 0) ? max(0, P - W + 1) : 0;
    const int n_cache_tiles = (P - lo + kTileKeys - 1) / kTileKeys;
    const int n_tiles = n_cache_tiles + 1;

    auto issue_tile = [&](int t, int buf) {
        const int start = (t < n_cache_tiles) ? lo + t * kTileKeys : P;
        const int count = (t < n_cache_tiles) ? min(kTileKeys, P - start) : n;
        uint8_t* base = raw_s + buf * S::kRawTile;
        constexpr int CPR = KB / 16;  // 16-byte chunks per code row
        for (int idx = tid; idx < count * CPR; idx += nthreads) {
            const int c = idx / CPR, ch = idx % CPR;
            const size_t g = (plane_row0 + start + c) * KB + ch * 16;
            cp_async16(base + c * KB + ch * 16, kq + g);
            cp_async16(base + S::kRawCodes + c * KB + ch * 16, vq + g);
        }
        // scale rows: NB halves = 2*NB bytes each (4, 8 or 16: one cp.async per row)
        uint8_t* ksd = base + 2 * S::kRawCodes;
        uint8_t* vsd = ksd + S::kRawScales;
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

    // First cache tile in flight before the tree rows are quantised (cache
    // tiles never touch slots >= P).
    int t_cur = rank;
    if (t_cur < n_cache_tiles) issue_tile(t_cur, 0);

    // Quantise this CTA's share of the tree rows (rows rank, rank + CS, ...)
    // of K and V into slots P + row; every cluster writes identical bytes.
    {
        const int mine = (n > rank) ? (n - rank + CS - 1) / CS : 0;
        for (int item = tid; item < mine * 2 * NB; item += nthreads) {
            const int j = item / (2 * NB), which = (item / NB) % 2, blk = item % NB;
            const int row = rank + CS * j;
            const uint16_t* src = (which ? a.v_new : a.k_new) + (((size_t)b * N + row) * a.Hkv + kvh) * D + blk * 32;
            const size_t slot = plane_row0 + P + row;
            uint8_t* codes = (which ? vq : kq) + slot * KB + blk * (KB / NB);
            uint16_t* sc = (which ? a.vs : a.ks) + slot * NB + blk;
            quantize_block<TYPE>(src, codes, sc);
        }
    }
    if (!block_tree_topology(a.parent + (size_t)b * N, n, N, par_s, depth_s, amask_s,
                             (rank == 0 && rt == 0 && kvh == 0) ? a.status : nullptr)) {
        cp_async_wait<0>();
        return;  // uniform over the cluster: the parent array is shared
    }
    __threadfence();
    cluster_sync_all();  // tree slots written by the whole cluster are now visible
    if (t_cur >= n_cache_tiles) {
        if (t_cur < n_tiles) issue_tile(t_cur, 0);
        else cp_async_commit();
    }

    // Query rows of this tile: row r <-> flat (node i, head gh) = row0 + r = i * G + gh, fp16.
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
        *reinterpret_cast<uint4*>(Q_s + r * HS + c8 * 8) = outv;
    }

    // Per-thread row metadata: rows gq and gq + 8 of this warp.
    int lb[2], rdepth[2];
    uint64_t ramask[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int rho = row0 + warp * 16 + gq + 8 * s;
        if (rho < rows_valid) {
            const int i = rho / G;
            rdepth[s] = depth_s[i];
            ramask[s] = amask_s[i];
            lb[s] = (W > 0) ? P + depth_s[i] - W + 1 : INT_MIN;
        } else {
            rdepth[s] = 0;
            ramask[s] = 0;
            lb[s] = INT_MAX;
        }
    }

    // ldmatrix lane addresses (bytes): Q as the A operand (rows x dims),
    // K rows as the B operand (keys x dims, non-transposed), V rows as the
    // B operand of p . V (keys x dims, transposed).
    const uint32_t q_addr = smem_u32(Q_s + (warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * HS + (lane >> 4) * 8);
    const uint32_t k_addr = smem_u32(Kh_s + ((lane & 7) + ((lane >> 4) & 1) * 8) * HS + ((lane >> 3) & 1) * 8);
    const uint32_t v_addr = smem_u32(Vh_s + ((lane & 7) + ((lane >> 3) & 1) * 8) * HS + (lane >> 4) * 8);

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
        const uint8_t* rb = raw_s + buf * S::kRawTile;
        const uint16_t* ksb = reinterpret_cast<const uint16_t*>(rb + 2 * S::kRawCodes);
        const uint16_t* vsb = reinterpret_cast<const uint16_t*>(rb + 2 * S::kRawCodes + S::kRawScales);

        // stage codes as exact fp16 integers (rows past count are zero) and
        // the block scales transposed to [block][key] in fp32
        for (int idx = tid; idx < 2 * kTileKeys * (D / 8); idx += nthreads) {
            const int which = idx / (kTileKeys * (D / 8));
            const int rem = idx % (kTileKeys * (D / 8));
            const int c = rem / (D / 8), d8 = rem % (D / 8);
            const uint8_t* src = rb + which * S::kRawCodes + c * KB;
            uint4 o = make_uint4(0, 0, 0, 0);
            if (c < count) {
                if constexpr (TYPE == DFLV_KV_Q8_0) {
                    const uint2 w = *reinterpret_cast<const uint2*>(src + d8 * 8);
                    i8x4_to_f16x2(w.x, o.x, o.y);
                    i8x4_to_f16x2(w.y, o.z, o.w);
                } else {
                    // dims d8*8 .. +7 of 32-block blk: low (first half of the
                    // block) or high nibbles of 8 consecutive bytes
                    const int blk = (d8 * 8) / 32, off = (d8 * 8) % 32;
                    const uint2 w = *reinterpret_cast<const uint2*>(src + blk * 16 + (off & 15));
                    const int sh = off >= 16 ? 4 : 0;
                    u4x4_to_f16x2((w.x >> sh) & 0x0f0f0f0fu, o.x, o.y);
                    u4x4_to_f16x2((w.y >> sh) & 0x0f0f0f0fu, o.z, o.w);
                }
            }
            *reinterpret_cast<uint4*>((which ? Vh_s : Kh_s) + c * HS + d8 * 8) = o;
        }
        for (int idx = tid; idx < 2 * NB * kTileKeys; idx += nthreads) {
            const int which = idx / (NB * kTileKeys), rem = idx % (NB * kTileKeys);
            const int blk = rem / kTileKeys, c = rem % kTileKeys;
            const uint16_t* sb = which ? vsb : ksb;
            (which ? VsT_s : KsT_s)[rem] = (c < count) ? __half2float(__ushort_as_half(sb[c * NB + blk])) : 0.f;
        }
        __syncthreads();

        // scores: S = sum over 32-dim blocks of d_k * (q . codes), on tensor cores
        float Sacc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) Sacc[nt][0] = Sacc[nt][1] = Sacc[nt][2] = Sacc[nt][3] = 0.f;
#pragma unroll 2
        for (int blk = 0; blk < NB; ++blk) {
            uint32_t qa[2][4];
            ldmatrix_x4(qa[0], q_addr + (2 * blk) * 32);
            ldmatrix_x4(qa[1], q_addr + (2 * blk + 1) * 32);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t kb0[4], kb1[4];
                ldmatrix_x4(kb0, k_addr + np * 16 * HS * 2 + (2 * blk) * 32);
                ldmatrix_x4(kb1, k_addr + np * 16 * HS * 2 + (2 * blk + 1) * 32);
                float tA[4] = {0.f, 0.f, 0.f, 0.f}, tB[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t bA0[2] = {kb0[0], kb0[1]}, bA1[2] = {kb1[0], kb1[1]};
                const uint32_t bB0[2] = {kb0[2], kb0[3]}, bB1[2] = {kb1[2], kb1[3]};
                mma_f16_16816(tA, qa[0], bA0);
                mma_f16_16816(tA, qa[1], bA1);
                mma_f16_16816(tB, qa[0], bB0);
                mma_f16_16816(tB, qa[1], bB1);
                const float2 sA = *reinterpret_cast<const float2*>(KsT_s + blk * kTileKeys + np * 16 + tq * 2);
                const float2 sB = *reinterpret_cast<const float2*>(KsT_s + blk * kTileKeys + np * 16 + 8 + tq * 2);
                Sacc[2 * np][0] = fmaf(tA[0], sA.x, Sacc[2 * np][0]);
                Sacc[2 * np][1] = fmaf(tA[1], sA.y, Sacc[2 * np][1]);
                Sacc[2 * np][2] = fmaf(tA[2], sA.x, Sacc[2 * np][2]);
                Sacc[2 * np][3] = fmaf(tA[3], sA.y, Sacc[2 * np][3]);
                Sacc[2 * np + 1][0] = fmaf(tB[0], sB.x, Sacc[2 * np + 1][0]);
                Sacc[2 * np + 1][1] = fmaf(tB[1], sB.y, Sacc[2 * np + 1][1]);
                Sacc[2 * np + 1][2] = fmaf(tB[2], sB.x, Sacc[2 * np + 1][2]);
                Sacc[2 * np + 1][3] = fmaf(tB[3], sB.y, Sacc[2 * np + 1][3]);
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
        // The running max only moves when a row's tile max exceeds it by more
        // than 2^8 (log2 domain): weights stay <= 256, exact after the final
        // normalisation, and O is rescaled only on those (rare) tiles.
        float alpha[2];
        bool rescale = false;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            mt[s] = fmaxf(mt[s], __shfl_xor_sync(0xffffffffu, mt[s], 1));
            mt[s] = fmaxf(mt[s], __shfl_xor_sync(0xffffffffu, mt[s], 2));
            alpha[s] = 1.f;
            if (mt[s] > m_run[s] + 8.f) {
                alpha[s] = (m_run[s] == -INFINITY) ? 0.f : exp2f(m_run[s] - mt[s]);
                m_run[s] = mt[s];
                l_run[s] *= alpha[s];
                rescale = true;
            }
            mt[s] = (m_run[s] == -INFINITY) ? 0.f : m_run[s];
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
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int j = 0; j < D / 8; ++j) {
                O[j][0] *= alpha[0];
                O[j][1] *= alpha[0];
                O[j][2] *= alpha[1];
                O[j][3] *= alpha[1];
            }
        }

        // O += (P * d_v) V_codes on tensor cores, one 32-dim V block at a time
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
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
                    ldmatrix_x4_trans(r, v_addr + kk * 16 * HS * 2 + dn * 32);
                    const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
                    mma_f16_16816(O[2 * dn], pa, b0);
                    mma_f16_16816(O[2 * dn + 1], pa, b1);
                }
            }
        }
        __syncthreads();  // staged tile consumed: the next one may overwrite it
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
    grid_launch_dependents();
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
    int RT, n_rt;
};

RowTiling choose_rows(const AttnVerifyArgs& a) {
    const int rows = (a.Hq / a.Hkv) * a.N_max;
    RowTiling t;
    t.n_rt = (rows + kMaxRowTile - 1) / kMaxRowTile;
    const int per = (rows + t.n_rt - 1) / t.n_rt;
    t.RT = ((per + 15) / 16) * 16;
    return t;
}

// Largest cluster (power of two, <= 16) that the SMs can hold at one CTA per
// SM alongside the others and that the key range can feed; 16 uses the
// non-portable cluster size when the device can schedule it.
template <typename Kernel>
int choose_cluster(Kernel kern, const AttnVerifyArgs& a, const RowTiling& t, size_t smem, int sms) {
    const long range = (a.window > 0) ? (long)a.window - 1 : (long)a.cap;
    const long tiles = (range + kTileKeys - 1) / kTileKeys + 1;
    const long clusters = (long)t.n_rt * a.Hkv * a.B;
    int cs = 1;
    while (cs < 8 && clusters * cs * 2 <= sms && cs * 2 <= tiles) cs *= 2;
    if (cs == 16) {
        static int ok16 = -1;  // probed once per process
        if (ok16 < 0) {
            ok16 = 0;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(16, 1, 1);
                cfg.blockDim = dim3(t.RT * 2, 1, 1);
                cfg.dynamicSmemBytes = smem;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 16;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n_clusters = 0;
                if (cudaOccupancyMaxActiveClusters(&n_clusters, kern, &cfg) == cudaSuccess && n_clusters >= 1)
                    ok16 = 1;
            }
            cudaGetLastError();
        }
        if (!ok16) cs = 8;
    }
    return cs;
}

template <int D, int TYPE>
cudaError_t launch_main(const AttnVerifyArgs& a, cudaStream_t stream) {
    using S = AttnSmem<D, TYPE>;
    const RowTiling t = choose_rows(a);
    const size_t smem = S::total(t.RT);
    auto kern = attn_tree_verify_kernel<D, TYPE>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const int cs = choose_cluster(kern, a, t, smem, sm_count_cached());
    return launch_pdl(kern, dim3(cs, t.n_rt * a.Hkv, a.B), dim3(t.RT * 2), smem, stream, cs, a, t.RT, cs);
}

}  // namespace

size_t attn_workspace_bytes(const AttnVerifyArgs& a) {
    if (a.type == DFLV_KV_F32) return 0;
    return (a.D == 128 || a.D == 256) ? attn_workspace_bytes_tc(a) : 0;
}

cudaError_t launch_attn_tree_verify(const AttnVerifyArgs& a, cudaStream_t stream) {
    if (a.type == DFLV_KV_F32) {
        cudaError_t e = launch_pdl(attn_store_tree_f32_kernel, dim3(a.N_max, a.Hkv, a.B), dim3(64), 0, stream, 1, a);
        if (e != cudaSuccess) return e;
        return launch_pdl(attn_tree_verify_f32_kernel, dim3((a.N_max + 7) / 8, a.Hq, a.B), dim3(256), 0, stream, 1, a);
    }
    // head sizes 128 / 256: the tensor-memory kernel (attn_verify_tc.cu);
    // 64: the warp-MMA kernel below
    if (a.D == 128 || a.D == 256) return launch_attn_tree_verify_tc(a, stream);
    const bool q8 = a.type == DFLV_KV_Q8_0;
    if (a.D == 64) return q8 ? launch_main<64, DFLV_KV_Q8_0>(a, stream) : launch_main<64, DFLV_KV_Q4_0>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace dflv
