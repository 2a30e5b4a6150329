// fwd_kernel.cuh -- exact ring-attention forward for sm_103a.
//
// What it computes ("Training Long-Context Models Without OOM: Ring
// Attention", section "Ring Attention Demystified", steps 1-5; "Context
// Parallelism" guide, section 2 "How It Works"):  the sequence of one
// (batch, head) is split into P equal contiguous chunks of C = S / P rows.
// Query chunk i visits KV chunk j = (i - t) mod P at ring step t = 0..P-1
// (step 0 is its own chunk, later steps the left neighbour's); causal
// attention skips chunks j > i and masks key > query inside chunk i.  Every
// visit updates running softmax statistics -- the row maximum and the sum of
// exponentials -- so the result equals unchunked attention:
//     O_r = sum_c exp(s_rc - LSE_r) v_c,   LSE_r = ln sum_c exp(s_rc).
//
// On one GPU the P "ranks" are chunks and the ring rotation becomes the TMA
// producer streaming K/V tiles of chunk j, then j-1, ... through a ring of
// shared-memory stages, so the next tile (and the first tile of the next
// chunk) is in flight while the current one is multiplied -- the
// single-device counterpart of "communication of K/V rotation overlapped
// with the attention computation of the current step" (guide, section 2,
// "Communication").
//
// CTA layout (320 threads):
//   warp 0      TMA producer: Q tiles once, then K/V tiles in ring order.
//   warp 1      TMEM allocator and MMA issuer (converged; elect.sync picks the issuing lane).
//   warps 2-5   softmax / epilogue for query tile 0 (rows 0..127).
//   warps 6-9   softmax / epilogue for query tile 1 (rows 128..255).
// The two query tiles share every K/V tile.  TMEM (512 columns):
//   [0,128) S0 / P0, [128,256) S1 / P1, [256,256+D) O0, [256+D,256+2D) O1.
// P (bf16) is written over the first 64 columns of its S and fed to the
// P.V MMA straight from TMEM; tcgen05 MMAs of one CTA run in issue order,
// so the next S = Q K^T (issued after P.V) cannot overwrite P early.
//
// Q, K and V are read through tensor maps built from the caller's row
// layout (layout.cuh) -- 3-D {d, S, B * H} when batch and head fold into
// one index, else 4-D {d, S, H, B} -- so [B, H, S, d], [B, S, H, d] and
// other layouts with contiguous d-element rows share one code path; O is
// stored through the same kind of layout.
//
// Online softmax: scores are taken in the log2 domain (x = s * scale *
// log2 e).  The running maximum used for exponentiation is only raised when
// the row maximum exceeds it by more than 8 (a factor 256); otherwise the
// stale maximum is kept.  O and l always share the same reference, so the
// final O / l and LSE = (m + log2 l) ln 2 are exact; only the rescale work
// is saved.
#pragma once

#include "layout.cuh"
#include "sm103_ptx.cuh"
#include "trace.cuh"

namespace ra {
namespace fwd {

constexpr int kBM = 128;      // query rows per tile
constexpr int kBN = 128;      // keys per KV tile
constexpr int kQTiles = 2;    // query tiles per CTA
constexpr int kRowsPerCta = kBM * kQTiles;
constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static constexpr int kBoxes = D / 64;                       // 64-col TMA boxes per tile
    static constexpr int kBoxBytes = 64 * kBN * 2;              // 16 KB
    static constexpr int kTileBytes = kBN * D * 2;              // one Q, K or V tile
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQTiles * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;   // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;          // S_u at kColS + 128 u
    static constexpr uint32_t kColO = 256;        // O_u at kColO + D u
};

struct FwdParams {
    __nv_bfloat16* o;       // [B, H, S, D] rows placed by `lo`
    RowLayout lo;
    int rank4;              // bit set: the q (1), k (2), v (4) map is 4-D
    float* lse;             // [B, H, S]
    int S, P, C;            // sequence, chunks, chunk length
    int H, group;           // query heads; query heads per key/value head
    // Emulated ring (one step at a time): step >= 0 restricts the CTA to KV
    // chunk j = (i - step) mod P, read from rank i's receive buffer -- a
    // [P * B * H, C, D] tensor whose head index is i * BH + bh -- and writes
    // the normalized partial O in fp32 to o32.  step = -1 is the fused ring.
    int step, BH;
    float* o32;
    int causal;
    int pairs_per_chunk;    // ceil(C / 256)
    float scale_log2;       // scale * log2(e)
    uint32_t* status;
    uint64_t wait_limit_ns;
};

// Ring-ordered sequence of KV tiles of one CTA.  Chunk j = i, i-1, ... (mod
// P); causal drops j > i.  Inside chunk i (causal) only tiles holding keys
// <= the CTA's last query row are visited.
struct RingTiles {
    int P, C, i, causal, tiles_per_chunk, tiles_local;
    int t, j, kt, kt_count;

    __device__ __forceinline__ void init(int P_, int C_, int i_, int causal_, int q_last_excl)
    {
        P = P_; C = C_; i = i_; causal = causal_;
        tiles_per_chunk = (C + kBN - 1) / kBN;
        tiles_local = causal ? (q_last_excl - i * C + kBN - 1) / kBN : tiles_per_chunk;
        t = 0; j = i; kt = 0; kt_count = tiles_local;
    }
    // One ring step only: chunk j = (i - t) mod P; nothing when causal and
    // j > i.
    __device__ __forceinline__ void init_step(int P_, int C_, int i_, int t_, int causal_, int q_last_excl)
    {
        P = P_; C = C_; i = i_; causal = causal_;
        tiles_per_chunk = (C + kBN - 1) / kBN;
        t = t_;
        j = ((i - t) % P + P) % P;
        if (causal && j > i)
            kt_count = 0;
        else if (causal && j == i)
            kt_count = (q_last_excl - i * C + kBN - 1) / kBN;
        else
            kt_count = tiles_per_chunk;
        tiles_local = kt_count;
        kt = 0;
    }
    __device__ __forceinline__ int total() const
    {
        return causal ? tiles_local + i * tiles_per_chunk : P * tiles_per_chunk;
    }
    __device__ __forceinline__ int key_start() const { return j * C + kt * kBN; }
    __device__ __forceinline__ int chunk_end() const { return (j + 1) * C; }
    __device__ __forceinline__ void next()
    {
        if (++kt < kt_count) return;
        kt = 0;
        ++t;
        j = j == 0 ? P - 1 : j - 1;       // receive from the left neighbour
        kt_count = tiles_per_chunk;       // every later chunk is visited whole
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
ring_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const FwdParams p)
{
    using CF = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw_base);

    const uint32_t sQ = base + CF::kOffQ;
    const uint32_t sK = base + CF::kOffK;
    const uint32_t sV = base + CF::kOffV;
    const uint32_t bar0 = base + CF::kOffBar;
    // barrier slots (8 bytes each)
    const uint32_t bar_q = bar0;
    auto bar_k_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto bar_k_empty = [&](int s) { return bar0 + 8u * (1 + CF::kStages + s); };
    auto bar_v_full = [&](int s) { return bar0 + 8u * (1 + 2 * CF::kStages + s); };
    auto bar_v_empty = [&](int s) { return bar0 + 8u * (1 + 3 * CF::kStages + s); };
    const uint32_t bar_misc = bar0 + 8u * (1 + 4 * CF::kStages);
    auto bar_s_full = [&](int u) { return bar_misc + 8u * u; };          // MMA -> softmax
    auto bar_p_full = [&](int u) { return bar_misc + 8u * (2 + u); };    // softmax -> MMA
    const uint32_t bar_o_final = bar_misc + 8u * 4;                      // last P.V done
    const uint32_t bar_drain = bar_misc + 8u * 5;                        // MMA drain at exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + CF::kOffBar + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + CF::kOffBar + 200);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: (b*H + h, query chunk i, pair u), heaviest first -----
    const int items_per_head = p.P * p.pairs_per_chunk;
    const int bh = blockIdx.x / items_per_head;
    const int g = items_per_head - 1 - (blockIdx.x % items_per_head);
    const int chunk_i = g / p.pairs_per_chunk;
    const int q0 = chunk_i * p.C + (g % p.pairs_per_chunk) * kRowsPerCta;
    const int q_end = min(q0 + kRowsPerCta, (chunk_i + 1) * p.C);   // rows stored
    // key/value head of this query head (grouped-query attention: query
    // head h reads key/value head h / group)

    WaitCtl wc{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int s = 0; s < CF::kStages; ++s) {
            mbar_init(bar_k_full(s), 1);
            mbar_init(bar_k_empty(s), 1);
            mbar_init(bar_v_full(s), 1);
            mbar_init(bar_v_empty(s), 1);
        }
        for (int u = 0; u < kQTiles; ++u) {
            mbar_init(bar_s_full(u), 1);
            mbar_init(bar_p_full(u), kBM);
        }
        mbar_init(bar_o_final, 1);
        mbar_init(bar_drain, 1);
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

    const bool step_mode = p.step >= 0;
    RingTiles rt;
    int NT;
    if (step_mode) {
        rt.init_step(p.P, p.C, chunk_i, p.step, p.causal, q_end);
        NT = rt.kt_count;
    } else {
        rt.init(p.P, p.C, chunk_i, p.causal, q_end);
        NT = rt.total();
    }
    // K/V rows are relative to the chunk start in step mode.
    const int kv_row0 = step_mode ? rt.j * p.C : 0;

    if (NT == 0) {
        // Nothing to attend to in this ring step (causal, chunk above the
        // diagonal): the partial is the merge identity, O = 0, LSE = -inf.
        if (threadIdx.x == 0) {
            int* tr = trace_slot(p.P);
            if (tr) trace_put(tr, bh, chunk_i, q0, 0, p.step, 0);
        }
        if (warp >= 2) {
            const int u = (warp - 2) >> 2;
            const int row = q0 + kBM * u + (warp & 3) * 32 + lane;
            if (row < q_end && p.o32) {
                float4* dst = reinterpret_cast<float4*>(p.o32 + ((size_t)bh * p.S + row) * D);
#pragma unroll
                for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.lse[(size_t)bh * p.S + row] = -INFINITY;
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            // batch and head of this CTA; K/V come from the key/value head
            // of the fused ring, or from this rank's receive buffer -- a
            // [P * B, H, C, D] tensor, rows relative to the chunk start -- in
            // step mode
            const int b_idx = bh / p.H;
            const int h_idx = bh - b_idx * p.H;
            const int kv_h = step_mode ? h_idx : h_idx / p.group;
            const int kv_b = step_mode ? chunk_i * (p.BH / p.H) + b_idx : b_idx;
            const int kv_heads = step_mode ? p.H : p.H / p.group;
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            mbar_arrive_expect_tx(bar_q, kQTiles * CF::kTileBytes);
            for (int u = 0; u < kQTiles; ++u)
                for (int x = 0; x < CF::kBoxes; ++x)
                    tma_load_rows(sQ + u * CF::kTileBytes + x * CF::kBoxBytes, &map_q, bar_q,
                                  64 * x, q0 + kBM * u, h_idx, b_idx, p.H, (p.rank4 & 1) != 0);
            int issued_k[CF::kStages], issued_v[CF::kStages];
            for (int s = 0; s < CF::kStages; ++s) issued_k[s] = issued_v[s] = -1;
            bool ok = true;
            int* tr = trace_slot(p.P);   // NULL unless the visit order is being recorded
            int visits = 0;
            for (int n = 0; n < NT && ok; ++n, rt.next()) {
                const int s = n % CF::kStages;
                const uint32_t ph = (uint32_t)(n / CF::kStages) & 1u;
                const int key0 = rt.key_start();
                if (tr && rt.kt == 0 && visits < p.P) {   // the stream enters chunk j
                    ++visits;
                    trace_put(tr + visits * kTraceInts, rt.t, rt.j, rt.j == chunk_i ? 0 : 1, rt.kt_count, key0,
                              key0 + (rt.kt_count - 1) * kBN);
                }
                ok = mbar_wait(bar_k_empty(s), ph ^ 1u, wc);
                if (!ok) break;
                mbar_arrive_expect_tx(bar_k_full(s), CF::kTileBytes);
                for (int x = 0; x < CF::kBoxes; ++x)
                    tma_load_rows(sK + s * CF::kTileBytes + x * CF::kBoxBytes, &map_k,
                                  bar_k_full(s), 64 * x, key0 - kv_row0, kv_h, kv_b, kv_heads, (p.rank4 & 2) != 0);
                issued_k[s] = (int)ph;
                ok = mbar_wait(bar_v_empty(s), ph ^ 1u, wc);
                if (!ok) break;
                mbar_arrive_expect_tx(bar_v_full(s), CF::kTileBytes);
                for (int x = 0; x < CF::kBoxes; ++x)
                    tma_load_rows(sV + s * CF::kTileBytes + x * CF::kBoxBytes, &map_v,
                                  bar_v_full(s), 64 * x, key0 - kv_row0, kv_h, kv_b, kv_heads, (p.rank4 & 4) != 0);
                issued_v[s] = (int)ph;
            }
            if (tr) trace_put(tr, bh, chunk_i, q0, visits, p.step, NT);
            if (!ok) {
                // Let every copy still in flight land before the CTA exits.
                WaitCtl drain{abort_flag, p.status, 200000000ull};
                volatile int dummy = 0;
                drain.abort_flag = &dummy;
                mbar_wait(bar_q, 0, drain);
                for (int s = 0; s < CF::kStages; ++s) {
                    if (issued_k[s] >= 0) mbar_wait(bar_k_full(s), (uint32_t)issued_k[s], drain);
                    if (issued_v[s] >= 0) mbar_wait(bar_v_full(s), (uint32_t)issued_v[s], drain);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        // The whole warp runs this loop converged and waits together; one
        // elected lane issues each group of MMAs and the commits.  The SM
        // takes one tcgen05.mma about every 48 cycles against 64 cycles of
        // work for a 128x128x16 step, so the issuing thread has little slack:
        // keeping the operands warp-uniform keeps the code around each MMA
        // short.
        {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, false, true);
            // Descriptor bases; a k-step only moves the start address -- the
            // descriptor's low field, address / 16 -- by a constant.
            const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sV, CF::kBoxBytes, 1024);
            constexpr uint32_t kTile16 = CF::kTileBytes >> 4;
            auto issue_s = [&](int u, int s) {
                const uint32_t d_tmem = tmem + CF::kColS + 128u * u;
                const uint64_t dq = dq0 + (uint32_t)u * kTile16;
                const uint64_t dk = dk0 + (uint32_t)s * kTile16;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        constexpr uint32_t kBox16 = CF::kBoxBytes >> 4;
                        const uint32_t off16 = (kk >> 2) * kBox16 + (kk & 3) * 2;
                        mma_bf16_ss(d_tmem, dq + off16, dk + off16, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                }
                __syncwarp();
            };
            auto issue_pv = [&](int u, int s, bool first) {
                const uint32_t d_tmem = tmem + CF::kColO + (uint32_t)D * u;
                const uint32_t a_tmem = tmem + CF::kColS + 128u * u;
                const uint64_t dv = dv0 + (uint32_t)s * kTile16;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_bf16_ts(d_tmem, a_tmem + 8u * kk, dv + (uint32_t)kk * (2048 >> 4), idesc_pv,
                                    (first && kk == 0) ? 0u : 1u);
                }
                __syncwarp();
            };
            // elect.sync picks the lowest lane every time, so the commits come
            // from the thread that issued the MMAs they track.
            auto commit = [&](uint32_t bar) {
                if (elect_one()) mma_commit(bar);
                __syncwarp();
            };
            auto wait_all = [&](uint32_t bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
            };
            bool ok = wait_all(bar_q, 0) && wait_all(bar_k_full(0), 0);
            if (ok) {
                tc_fence_after();
                for (int u = 0; u < kQTiles; ++u) {
                    issue_s(u, 0);
                    commit(bar_s_full(u));
                }
                commit(bar_k_empty(0));
            }
            for (int n = 0; n < NT && ok; ++n) {
                const int s = n % CF::kStages;
                const uint32_t ph = (uint32_t)(n / CF::kStages) & 1u;
                const int s1 = (n + 1) % CF::kStages;
                const uint32_t ph1 = (uint32_t)((n + 1) / CF::kStages) & 1u;
                const bool more = n + 1 < NT;
                ok = wait_all(bar_v_full(s), ph);
                if (!ok) break;
                for (int u = 0; u < kQTiles && ok; ++u) {
                    ok = wait_all(bar_p_full(u), (uint32_t)n & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(u, s, n == 0);
                    if (u == kQTiles - 1) commit(bar_v_empty(s));
                    if (more) {
                        if (u == 0) {
                            ok = wait_all(bar_k_full(s1), ph1);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        issue_s(u, s1);
                        commit(bar_s_full(u));
                        if (u == kQTiles - 1) commit(bar_k_empty(s1));
                    }
                }
            }
            if (ok) commit(bar_o_final);
            // Every MMA issued so far must finish before TMEM is released.
            commit(bar_drain);
            WaitCtl drain{abort_flag, p.status, 200000000ull};
            volatile int dummy = 0;
            drain.abort_flag = &dummy;
            __all_sync(0xffffffffu, mbar_wait(bar_drain, 0, drain));
        }
    } else {
        // ------------------------------------------------ softmax + epilogue
        const int u = (warp - 2) >> 2;                 // query tile 0 or 1
        const uint32_t quarter = (uint32_t)(warp & 3); // TMEM lane quarter
        const int r = (int)quarter * 32 + lane;        // row inside the tile
        const int row = q0 + kBM * u + r;              // position in the head
        const uint32_t tS = tmem_addr(tmem, quarter * 32, CF::kColS + 128u * u);
        const uint32_t tO = tmem_addr(tmem, quarter * 32, CF::kColO + (uint32_t)D * u);
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY;   // running maximum (log2 domain)
        float l = 0.f;              // running sum of 2^(x - m_used)
        bool ok = true;
        for (int n = 0; n < NT; ++n, rt.next()) {
            // all lanes leave together: the tcgen05 loads below are warp-wide
            ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full(u), (uint32_t)n & 1u, wc));
            if (!ok) break;
            tc_fence_after();
            uint32_t s[128];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                tmem_ld32(tS + 32u * c4, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c4]));
            }
            tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[0]));
            tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[32]));
            tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[64]));
            tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[96]));
            const int key0 = rt.key_start();
            const int kend = rt.chunk_end();
            const bool local = rt.j == chunk_i;   // the query chunk's own KV chunk
            // Masking is needed on a tile that runs past its chunk's end or,
            // causal, on the local chunk's tiles that reach above row q0+128u.
            const bool need_mask = (key0 + kBN > kend) ||
                                   (p.causal && local && key0 + kBN - 1 > q0 + kBM * u);
            if (need_mask) {
                const int lim_causal = (p.causal && local) ? row - key0 : kBN;
                const int lim = min(kend - key0 - 1, lim_causal);   // last allowed column
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > lim) s[c] = __float_as_uint(-INFINITY);
            }
            // Row maximum: four independent chains of 3-input maxima.
            float mq[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) mq[a] = __uint_as_float(s[a]);
#pragma unroll
            for (int c = 4; c < 124; c += 8) {
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    mq[a] = max3f(mq[a], __uint_as_float(s[c + 2 * a]), __uint_as_float(s[c + 2 * a + 1]));
            }
            mq[0] = max3f(mq[0], __uint_as_float(s[124]), __uint_as_float(s[125]));
            mq[1] = max3f(mq[1], __uint_as_float(s[126]), __uint_as_float(s[127]));
            const float mx = max3f(mq[0], mq[1], fmaxf(mq[2], mq[3]));
            const float m_new = mx * sl2;
            const bool raise = m_new > m_used + kRescaleThreshold;
            float alpha = 1.f;
            if (raise) {
                alpha = ex2_approx(m_used - m_new);   // 0 when m_used = -inf
                m_used = m_new;
            }
            const float mb = (m_used == -INFINITY) ? 0.f : m_used;
            // p = 2^(s * scale * log2 e - m); the row sum in four partials.
            float sp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
                const float p0 = ex2_approx(fmaf(__uint_as_float(s[c]), sl2, -mb));
                const float p1 = ex2_approx(fmaf(__uint_as_float(s[c + 1]), sl2, -mb));
                const int a = (c >> 1) & 1;
                sp[2 * a] += p0;
                sp[2 * a + 1] += p1;
                s[c >> 1] = pack_bf16x2(p0, p1);
            }
            const float sum = (sp[0] + sp[1]) + (sp[2] + sp[3]);
            tmem_st32(tS, *reinterpret_cast<const uint32_t(*)[32]>(&s[0]));
            tmem_st32(tS + 32u, *reinterpret_cast<const uint32_t(*)[32]>(&s[32]));
            l = l * alpha + sum;
            if (n > 0 && __any_sync(0xffffffffu, raise)) {
                // O_u is idle: the S_u just read was issued after the last
                // P_u.V, and its completion covers every earlier MMA.
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32u * c4, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tmem_st32(tO + 32u * c4, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p_full(u));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_o_final, 0, wc));
        if (ok) {
            tc_fence_after();
            const bool store = row < q_end;
            const float inv_l = 1.f / l;
            const int srow = store ? row : 0;
            const int b_idx = bh / p.H;
            const size_t orow_off = p.o32 ? ((size_t)bh * p.S + (size_t)srow) * D
                                          : p.lo.row(b_idx, bh - b_idx * p.H, srow);
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t o[32];
                tmem_ld32(tO + 32u * c4, o);
                tmem_ld_wait(o);
                if (p.o32) {
                    // partial of one ring step, fp32 for the merge
                    if (store) {
                        float4* dst = reinterpret_cast<float4*>(p.o32 + orow_off + 32 * c4);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            dst[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv_l,
                                                  __uint_as_float(o[4 * v4 + 1]) * inv_l,
                                                  __uint_as_float(o[4 * v4 + 2]) * inv_l,
                                                  __uint_as_float(o[4 * v4 + 3]) * inv_l);
                    }
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        pk[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l,
                                            __uint_as_float(o[2 * c + 1]) * inv_l);
                    if (store) {
                        uint4* dst = reinterpret_cast<uint4*>(p.o + orow_off + 32 * c4);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                }
            }
            if (store) p.lse[(size_t)bh * p.S + row] = (m_used + log2f(l)) * 0.69314718055994531f;
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

}  // namespace fwd
}  // namespace ra
