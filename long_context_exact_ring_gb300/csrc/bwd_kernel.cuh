// bwd_kernel.cuh -- exact ring-attention backward for sm_103a.
//
// The pages keep activations for the backward pass and recompute to trade
// compute for memory ("Training Long-Context Models Without OOM: Ring
// Attention", "Diagnosing the Sequence-Length OOM" and "Why the Parallelism
// You Already Have Will Not Work"); they print no backward formulas.  This is
// the plain derivative of O_r = sum_c exp(s_rc - LSE_r) v_c for the loss
// L = sum(dO * O), with the attention matrix recomputed from the saved LSE:
//     P_rc = exp(s_rc - LSE_r) on the allowed set (0 elsewhere)
//     dV = P^T dO,   dP = dO V^T,   D_r = sum_k dO_rk O_rk,
//     dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q.
//
// Schedule: one CTA owns one 128-key tile of KV chunk j (K and V stay in
// shared memory; dK and dV accumulate in TMEM) and streams the 128-row query
// tiles that meet chunk j in the ring: query chunk i = j, j+1, ... (mod P) --
// chunk j is visited by query chunk i at ring step t = (i - j) mod P.  Causal
// drops i < j and, inside chunk j, query tiles wholly above the diagonal.
//
// Per query tile, on the tensor core (all bf16 x bf16 -> fp32):
//   S^T  = K Q^T      [keys x queries]   -> TMEM S   (A = K, B = Q, K-major)
//   dP^T = V dO^T     [keys x queries]   -> TMEM dP  (A = V, B = dO, K-major)
//   dV  += P^T dO     [keys x d]          A = P^T (bf16, TMEM), B = dO (MN-major)
//   dK  += dS^T Q     [keys x d]          A = dS^T (bf16, TMEM), B = Q (MN-major)
//   dQ_t = dS K       [queries x d]       A = dS (smem, MN-major), B = K (MN-major)
// TMEM (512 columns): S [0,128), dP [128,256), dV [256,256+D), dK after it.
// P^T (bf16) overwrites S[0,64) and dS^T overwrites dP[0,64); the dQ tile
// lands in the free upper halves S[64,128) (d columns 0..63) and dP[64,128)
// (d columns 64..127), from where four drain warps move it into the fp32 dQ
// accumulator in global memory with vector reductions.
//
// CTA layout (448 threads):
//   warp 0       TMA producer (K, V once; Q and dO tiles in ring order).
//   warp 1       TMEM allocator and MMA issuer.
//   warps 2-9    softmax-gradient: thread = key row; warps 2-5 take query
//                columns 0..63, warps 6-9 columns 64..127; epilogue dV
//                (warps 2-5) and dK (warps 6-9).
//   warps 10-13  dQ drain: thread = query row.
#pragma once

#include "sm103_ptx.cuh"
#include "small_kernels.cuh"
#include "profile.cuh"

namespace ra {
namespace bwd {

constexpr int kBK = 128;        // keys per CTA
constexpr int kBQ = 128;        // queries per streamed tile
constexpr int kThreads = 448;

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = 64 * 128 * 2;          // 16 KB: 128 rows x 64 bf16
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kStages = 2;                       // Q / dO stages
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;
    static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
    static constexpr int kOffDS = kOffDO + kStages * kTileBytes;        // 128 x 128 bf16
    static constexpr int kOffRow = kOffDS + 2 * kBoxBytes;              // lse2 / D staging
    static constexpr int kOffBar = kOffRow + 2 * 2 * kBQ * 4;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = kOffBar + kBarBytes;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColDP = 128;
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 256 + D;
};

struct BwdParams {
    const float* lse2;      // [B*H*S] LSE * log2(e)
    const float* Dvec;      // [B*H*S]
    float* dq_acc;          // [B*H*S, D] fp32, pre-zeroed
    __nv_bfloat16* dk;      // [B*H*S, D]
    __nv_bfloat16* dv;
    int S, P, C, causal, tiles_per_chunk;
    float scale, scale_log2;
    uint32_t* status;
    uint64_t wait_limit_ns;
};

// Query tiles met by key tile kt of chunk j, in ring order: chunks
// i = j, j+1, ... (mod P), each chunk's tiles ascending; causal keeps
// i >= j and, in chunk j, tiles from kt on.
struct QTiles {
    int P, C, j, causal, T, kt;
    int i, qt, qt_first;
    __device__ __forceinline__ void init(int P_, int C_, int j_, int causal_, int T_, int kt_)
    {
        P = P_; C = C_; j = j_; causal = causal_; T = T_; kt = kt_;
        i = j;
        qt_first = causal ? kt : 0;
        qt = qt_first;
    }
    __device__ __forceinline__ int total() const
    {
        return causal ? (T - kt) + (P - 1 - j) * T : P * T;
    }
    __device__ __forceinline__ int q_start() const { return i * C + qt * kBQ; }
    __device__ __forceinline__ int chunk_end() const { return (i + 1) * C; }
    __device__ __forceinline__ void next()
    {
        if (++qt < T) return;
        qt = 0;
        i = (i + 1 == P) ? 0 : i + 1;    // the chunk that meets j one ring step later
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
ring_bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                const BwdParams p)
{
    using CF = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = smem_u32(smem);
    if (base & 1023u) {   // the swizzled operand layouts need 1 KB alignment
        if (threadIdx.x == 0) atomicOr(p.status, kStatusAborted);
        return;
    }
    const uint32_t sK = base + CF::kOffK;
    const uint32_t sV = base + CF::kOffV;
    const uint32_t sQ = base + CF::kOffQ;
    const uint32_t sDO = base + CF::kOffDO;
    const uint32_t sDS = base + CF::kOffDS;
    float* row_lse2 = reinterpret_cast<float*>(smem + CF::kOffRow);        // [2][128]
    float* row_D = reinterpret_cast<float*>(smem + CF::kOffRow + 2 * kBQ * 4);
    const uint32_t bar0 = base + CF::kOffBar;
    const uint32_t bar_kv = bar0;
    auto bar_qdo_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (3 + s); };
    const uint32_t bar_s_full = bar0 + 8u * 5;
    const uint32_t bar_dp_full = bar0 + 8u * 6;
    const uint32_t bar_p_ready = bar0 + 8u * 7;
    const uint32_t bar_ds_ready = bar0 + 8u * 8;
    const uint32_t bar_dq_full = bar0 + 8u * 9;
    const uint32_t bar_dq_free = bar0 + 8u * 10;
    const uint32_t bar_kv_final = bar0 + 8u * 11;
    const uint32_t bar_drain = bar0 + 8u * 12;
    const uint32_t bar_group = bar0 + 8u * 13;   // rendezvous of the 256 softmax threads
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + CF::kOffBar + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + CF::kOffBar + 200);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: (b*H + h, KV chunk j, key tile kt), heaviest first ----
    const int T = p.tiles_per_chunk;
    const int items_per_head = p.P * T;
    const int bh = blockIdx.x / items_per_head;
    const int w = blockIdx.x % items_per_head;
    const int chunk_j = w / T;
    const int kt = w % T;
    const int k0 = chunk_j * p.C + kt * kBK;             // first key of the tile
    const int k_end = (chunk_j + 1) * p.C;               // keys >= k_end are not ours

    WaitCtl wc{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar_kv, 1);
        for (int s = 0; s < CF::kStages; ++s) {
            mbar_init(bar_qdo_full(s), 1);
            mbar_init(bar_qdo_empty(s), 1);
        }
        mbar_init(bar_s_full, 1);
        mbar_init(bar_dp_full, 1);
        mbar_init(bar_p_ready, 256);
        mbar_init(bar_ds_ready, 256);
        mbar_init(bar_dq_full, 1);
        mbar_init(bar_dq_free, 128);
        mbar_init(bar_kv_final, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_group, 256);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), CF::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    QTiles qi;
    qi.init(p.P, p.C, chunk_j, p.causal, T, kt);
    const int NT = qi.total();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            tma_prefetch_desc(&map_do);
            mbar_arrive_expect_tx(bar_kv, 2 * CF::kTileBytes);
            for (int x = 0; x < CF::kBoxes; ++x) {
                tma_load_3d(sK + x * CF::kBoxBytes, &map_k, bar_kv, 64 * x, k0, bh);
                tma_load_3d(sV + x * CF::kBoxBytes, &map_v, bar_kv, 64 * x, k0, bh);
            }
            int issued[CF::kStages];
            for (int s = 0; s < CF::kStages; ++s) issued[s] = -1;
            bool ok = true;
            for (int n = 0; n < NT; ++n, qi.next()) {
                const int s = n % CF::kStages;
                const uint32_t ph = (uint32_t)(n / CF::kStages) & 1u;
                ok = mbar_wait(bar_qdo_empty(s), ph ^ 1u, wc);
                if (!ok) break;
                const int q0 = qi.q_start();
                mbar_arrive_expect_tx(bar_qdo_full(s), 2 * CF::kTileBytes);
                for (int x = 0; x < CF::kBoxes; ++x) {
                    tma_load_3d(sQ + s * CF::kTileBytes + x * CF::kBoxBytes, &map_q,
                                bar_qdo_full(s), 64 * x, q0, bh);
                    tma_load_3d(sDO + s * CF::kTileBytes + x * CF::kBoxBytes, &map_do,
                                bar_qdo_full(s), 64 * x, q0, bh);
                }
                issued[s] = (int)ph;
            }
            if (!ok) {
                WaitCtl drain{abort_flag, p.status, 200000000ull};
                volatile int dummy = 0;
                drain.abort_flag = &dummy;
                mbar_wait(bar_kv, 0, drain);
                for (int s = 0; s < CF::kStages; ++s)
                    if (issued[s] >= 0) mbar_wait(bar_qdo_full(s), (uint32_t)issued[s], drain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc_kq = idesc_bf16_f32(kBK, kBQ, false, false);   // S^T, dP^T
            constexpr uint32_t idesc_kd = idesc_bf16_f32(kBK, D, false, true);      // dV, dK
            constexpr uint32_t idesc_qd = idesc_bf16_f32(kBQ, 64, true, true);      // dQ halves
            // C = A(smem, K-major) * B(smem, K-major)^T over the head dim.
            auto mma_kmajor = [&](uint32_t d_tmem, uint32_t sa, uint32_t sb) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * CF::kBoxBytes + (kk & 3) * 32;
                    mma_bf16_ss(d_tmem, sdesc_sw128(sa + off, 16, 1024),
                                sdesc_sw128(sb + off, 16, 1024), idesc_kq, kk > 0 ? 1u : 0u);
                }
            };
            // C += A(TMEM bf16, keys x queries) * B(smem, queries x D, MN-major)
            auto mma_ts = [&](uint32_t d_tmem, uint32_t a_tmem, uint32_t sb, bool first) {
#pragma unroll
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    mma_bf16_ts(d_tmem, a_tmem + 8u * kk,
                                sdesc_sw128(sb + kk * 2048, CF::kBoxBytes, 1024), idesc_kd,
                                (first && kk == 0) ? 0u : 1u);
            };
            bool ok = mbar_wait(bar_kv, 0, wc);
            for (int n = 0; n < NT && ok; ++n) {
                const int s = n % CF::kStages;
                const uint32_t ph = (uint32_t)(n / CF::kStages) & 1u;
                const uint32_t par = (uint32_t)n & 1u;
                ok = mbar_wait(bar_qdo_full(s), ph, wc);
                if (ok && n > 0) ok = mbar_wait(bar_dq_free, par ^ 1u, wc);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qs = sQ + s * CF::kTileBytes;
                const uint32_t dos = sDO + s * CF::kTileBytes;
                mma_kmajor(tmem + CF::kColS, sK, qs);
                mma_commit(bar_s_full);
                mma_kmajor(tmem + CF::kColDP, sV, dos);
                mma_commit(bar_dp_full);
                ok = mbar_wait(bar_p_ready, par, wc);
                if (!ok) break;
                tc_fence_after();
                mma_ts(tmem + CF::kColDV, tmem + CF::kColS, dos, n == 0);
                ok = mbar_wait(bar_ds_ready, par, wc);
                if (!ok) break;
                tc_fence_after();
                mma_ts(tmem + CF::kColDK, tmem + CF::kColDP, qs, n == 0);
                // dQ tile = dS K: A is dS^T stored [key][query] (queries
                // contiguous, MN-major), B is the K tile (d contiguous).
#pragma unroll
                for (int h = 0; h < CF::kBoxes; ++h) {
                    const uint32_t d_tmem = tmem + (h == 0 ? CF::kColS : CF::kColDP) + 64u;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_ss(d_tmem, sdesc_sw128(sDS + kk * 2048, CF::kBoxBytes, 1024),
                                    sdesc_sw128(sK + h * CF::kBoxBytes + kk * 2048, CF::kBoxBytes, 1024),
                                    idesc_qd, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar_dq_full);
                mma_commit(bar_qdo_empty(s));
            }
            if (ok) mma_commit(bar_kv_final);
            mma_commit(bar_drain);
            WaitCtl drain{abort_flag, p.status, 200000000ull};
            volatile int dummy = 0;
            drain.abort_flag = &dummy;
            mbar_wait(bar_drain, 0, drain);
        }
    } else if (warp < 10) {
        // ------------------------------------ P^T, dS^T; epilogue dV / dK
        const int half = (warp - 2) >> 2;                // query columns [64 half, +64)
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int kr = (int)quarter * 32 + lane;         // key row in the tile
        const int kpos = k0 + kr;
        const bool key_ok = kpos < k_end;
        const int tid = threadIdx.x - 64;                // 0..255
        const uint32_t tS = tmem_addr(tmem, quarter * 32, CF::kColS + 64u * half);
        const uint32_t tDP = tmem_addr(tmem, quarter * 32, CF::kColDP + 64u * half);
        const uint32_t tPo = tmem_addr(tmem, quarter * 32, CF::kColS + 32u * half);
        const uint32_t tDSo = tmem_addr(tmem, quarter * 32, CF::kColDP + 32u * half);
        const float sl2 = p.scale_log2;
        bool ok = true;
        // Bounded rendezvous of the 256 softmax threads (an mbarrier used as a
        // barrier): a thread that gives up cannot leave the others waiting
        // forever.
        uint32_t group_phase = 0;
        auto group_sync = [&]() -> bool {
            mbar_arrive(bar_group);
            const bool r = __all_sync(0xffffffffu, mbar_wait(bar_group, group_phase & 1u, wc));
            ++group_phase;
            return r;
        };
        for (int n = 0; n < NT; ++n, qi.next()) {
            const int q0 = qi.q_start();
            const int q_end = qi.chunk_end();
            const int buf = n & 1;
            // Stage this tile's per-query LSE (base 2) and D.  Queries past
            // the chunk end get LSE = +inf, i.e. P = 0.
            {
                const int qq = tid & 127;
                const int qpos = q0 + qq;
                const bool valid = qpos < q_end;
                const size_t gi = (size_t)bh * p.S + (size_t)(valid ? qpos : 0);
                if (tid < 128)
                    row_lse2[buf * kBQ + qq] = valid ? p.lse2[gi] : INFINITY;
                else
                    row_D[buf * kBQ + qq] = valid ? p.Dvec[gi] : 0.f;
            }
            ok = group_sync();
            if (!ok) break;
            ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full, (uint32_t)n & 1u, wc));
            if (!ok) break;
            tc_fence_after();
            uint32_t sv[64];
            tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld32(tS + 32u, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            // Causal: in chunk j's own query tiles, mask query < key.
            const bool diag = p.causal && qi.i == chunk_j && q0 + kBQ - 1 >= k0 && q0 <= k0 + kBK - 1;
            const float* lse2 = row_lse2 + buf * kBQ + 64 * half;
            float pv[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float e = ex2_approx(fmaf(__uint_as_float(sv[c]), sl2, -lse2[c]));
                if (diag && q0 + 64 * half + c < kpos) e = 0.f;
                pv[c] = key_ok ? e : 0.f;
            }
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
            // Both halves must have read S before either writes P over it.
            ok = group_sync();
            if (!ok) break;
            tmem_st32(tPo, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p_ready);

            ok = __all_sync(0xffffffffu, mbar_wait(bar_dp_full, (uint32_t)n & 1u, wc));
            if (!ok) break;
            tc_fence_after();
            const float* Dq = row_D + buf * kBQ + 64 * half;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t dp[32];
                tmem_ld32(tDP + 32u * c2, dp);
                tmem_ld_wait(dp);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int x = 32 * c2 + 2 * c;
                    pk[16 * c2 + c] = pack_bf16x2(pv[x] * (__uint_as_float(dp[2 * c]) - Dq[x]),
                                                  pv[x + 1] * (__uint_as_float(dp[2 * c + 1]) - Dq[x + 1]));
                }
            }
            // dS to shared memory as [key][query] rows, 128-byte swizzle: 16-byte
            // chunk c of row kr sits at chunk position c ^ (kr & 7).
            uint8_t* ds_row = smem + CF::kOffDS + half * CF::kBoxBytes + kr * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(ds_row + ((c ^ (kr & 7)) << 4)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            fence_proxy_async_smem();
            ok = group_sync();
            if (!ok) break;
            tmem_st32(tDSo, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_ds_ready);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_kv_final, 0, wc));
        if (ok) {
            tc_fence_after();
            // warps 2-5 write dV, warps 6-9 write dK (times scale)
            const uint32_t tAcc = tmem_addr(tmem, quarter * 32, half == 0 ? CF::kColDV : CF::kColDK);
            const float mul = half == 0 ? 1.f : p.scale;
            __nv_bfloat16* out = (half == 0 ? p.dv : p.dk) +
                                 ((size_t)bh * p.S + (size_t)(key_ok ? kpos : 0)) * D;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t a[32];
                tmem_ld32(tAcc + 32u * c4, a);
                tmem_ld_wait(a);
                uint32_t o16[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    o16[c] = pack_bf16x2(__uint_as_float(a[2 * c]) * mul, __uint_as_float(a[2 * c + 1]) * mul);
                if (key_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(out + 32 * c4);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(o16[4 * v4], o16[4 * v4 + 1], o16[4 * v4 + 2], o16[4 * v4 + 3]);
                }
            }
        }
    } else {
        // -------------------------------------------------------- dQ drain
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int qr = (int)quarter * 32 + lane;         // query row in the tile
        const uint32_t tA = tmem_addr(tmem, quarter * 32, CF::kColS + 64u);
        const uint32_t tB = tmem_addr(tmem, quarter * 32, CF::kColDP + 64u);
        const float sc = p.scale;
        for (int n = 0; n < NT; ++n, qi.next()) {
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_dq_full, (uint32_t)n & 1u, wc));
            if (!ok) break;
            tc_fence_after();
            const int qpos = qi.q_start() + qr;
            const bool row_ok = qpos < qi.chunk_end();
            float* dst = p.dq_acc + ((size_t)bh * p.S + (size_t)(row_ok ? qpos : 0)) * D;
            uint32_t a[32], b[32];
            tmem_ld32(tA, a);
            tmem_ld32(tA + 32u, b);
            tmem_ld_wait(a);
            tmem_ld_wait(b);
            if constexpr (D == 64) {
                tc_fence_before();
                mbar_arrive(bar_dq_free);
            }
            if (row_ok) {
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    red_add_v4(dst + c, __uint_as_float(a[c]) * sc, __uint_as_float(a[c + 1]) * sc,
                               __uint_as_float(a[c + 2]) * sc, __uint_as_float(a[c + 3]) * sc);
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    red_add_v4(dst + 32 + c, __uint_as_float(b[c]) * sc, __uint_as_float(b[c + 1]) * sc,
                               __uint_as_float(b[c + 2]) * sc, __uint_as_float(b[c + 3]) * sc);
            }
            if constexpr (D == 128) {
                tmem_ld32(tB, a);
                tmem_ld32(tB + 32u, b);
                tmem_ld_wait(a);
                tmem_ld_wait(b);
                tc_fence_before();
                mbar_arrive(bar_dq_free);
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        red_add_v4(dst + 64 + c, __uint_as_float(a[c]) * sc, __uint_as_float(a[c + 1]) * sc,
                                   __uint_as_float(a[c + 2]) * sc, __uint_as_float(a[c + 3]) * sc);
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        red_add_v4(dst + 96 + c, __uint_as_float(b[c]) * sc, __uint_as_float(b[c + 1]) * sc,
                                   __uint_as_float(b[c + 2]) * sc, __uint_as_float(b[c + 3]) * sc);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, CF::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline size_t workspace_bytes(int B, int H, int S, int d)
{
    const size_t rows = (size_t)B * H * S;
    return align256(rows * d * 4) + 2 * align256(rows * 4);
}

inline cudaError_t configure_kernels()
{
    cudaError_t e = cudaFuncSetAttribute(ring_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<64>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(ring_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<128>::kSmemBytes);
    return e;
}

struct Launch {
    const void *q, *k, *v, *o, *dO;
    const float* lse;
    void *dq, *dk, *dv;
    int B, H, S, d, P, causal;
    float scale;
    void* workspace;
    uint32_t* status;
    int num_sms;
    uint64_t wait_limit_ns;
    cudaStream_t stream;
    int (*encode)(CUtensorMap*, const void*, int, int, int, int);
};

// Zero the dQ accumulator, compute D and LSE2, run the main kernel, convert
// dQ.  Returns 0, or -3 (RA_ERR_CUDA) with *err set.
inline int launch(const Launch& L, cudaError_t* err)
{
    const size_t rows = (size_t)L.B * L.H * L.S;
    uint8_t* ws = static_cast<uint8_t*>(L.workspace);
    float* dq_acc = reinterpret_cast<float*>(ws);
    float* Dvec = reinterpret_cast<float*>(ws + align256(rows * L.d * 4));
    float* lse2 = reinterpret_cast<float*>(ws + align256(rows * L.d * 4) + align256(rows * 4));
    cudaError_t e = cudaMemsetAsync(dq_acc, 0, rows * L.d * 4, L.stream);
    if (e != cudaSuccess) { *err = e; return -3; }
    long long blocks = ((long long)rows + 7) / 8;
    const long long cap = (long long)L.num_sms * 16;
    if (blocks > cap) blocks = cap;
    const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(L.o);
    const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(L.dO);
    {
        prof::Scope ps(prof::kBwdPrep, L.stream);
        if (L.d == 128)
            bwd_prep_kernel<128><<<(unsigned)blocks, 256, 0, L.stream>>>(o, dO, L.lse, Dvec, lse2, (long long)rows);
        else
            bwd_prep_kernel<64><<<(unsigned)blocks, 256, 0, L.stream>>>(o, dO, L.lse, Dvec, lse2, (long long)rows);
        ps.done();
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = e; return -3; }

    CUtensorMap mq, mk, mv, mdo;
    const int BH = L.B * L.H;
    if (L.encode(&mq, L.q, BH, L.S, L.d, kBQ) || L.encode(&mk, L.k, BH, L.S, L.d, kBK) ||
        L.encode(&mv, L.v, BH, L.S, L.d, kBK) || L.encode(&mdo, L.dO, BH, L.S, L.d, kBQ)) {
        *err = cudaErrorInvalidValue;
        return -3;
    }
    BwdParams prm;
    prm.lse2 = lse2;
    prm.Dvec = Dvec;
    prm.dq_acc = dq_acc;
    prm.dk = static_cast<__nv_bfloat16*>(L.dk);
    prm.dv = static_cast<__nv_bfloat16*>(L.dv);
    prm.S = L.S;
    prm.P = L.P;
    prm.C = L.S / L.P;
    prm.causal = L.causal;
    prm.tiles_per_chunk = (prm.C + kBK - 1) / kBK;
    prm.scale = L.scale;
    prm.scale_log2 = (float)((double)L.scale * 1.4426950408889634);
    prm.status = L.status;
    prm.wait_limit_ns = L.wait_limit_ns;
    const long long grid = (long long)BH * L.P * prm.tiles_per_chunk;
    {
        prof::Scope ps(prof::kBwdMain, L.stream);
        if (L.d == 128)
            ring_bwd_kernel<128><<<(unsigned)grid, kThreads, Cfg<128>::kSmemBytes, L.stream>>>(mq, mk, mv, mdo, prm);
        else
            ring_bwd_kernel<64><<<(unsigned)grid, kThreads, Cfg<64>::kSmemBytes, L.stream>>>(mq, mk, mv, mdo, prm);
        ps.done();
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = e; return -3; }
    const long long n8 = (long long)(rows * L.d / 8);
    long long cb = (n8 + 255) / 256;
    if (cb > cap) cb = cap;
    {
        prof::Scope ps(prof::kDqConvert, L.stream);
        dq_convert_kernel<<<(unsigned)cb, 256, 0, L.stream>>>(dq_acc, static_cast<__nv_bfloat16*>(L.dq), n8);
        ps.done();
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = e; return -3; }
    return 0;
}

}  // namespace bwd
}  // namespace ra
