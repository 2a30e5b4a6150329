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
// With grouped-query attention the CTA streams these tiles for every query
// head of its key/value head's group, one head after the other, so dK and dV
// collect the whole group in TMEM.
//
// Per query tile n, on the tensor core (bf16 x bf16 -> fp32), in issue order:
//   dP^T = V dO^T     [keys x queries]  -> TMEM dP   (A = V, B = dO, K-major)
//   dV  += P^T dO     [keys x d]         A = P^T (bf16 in TMEM), B = dO (MN-major)
//   S^T  = K Q^T      of tile n + 1     -> TMEM S    (A = K, B = Q, K-major)
//   dK  += dS^T Q     [keys x d]         A = dS^T (bf16 in TMEM), B = Q (MN-major)
//   dQ_t = dS K       [queries x d]     -> TMEM dP   A = dS (smem, MN-major), B = K (MN-major)
// (S^T of the first tile is issued before the loop.)  TMEM (512 columns):
// S [0,128), dP [128,256), dV [256,256+D), dK after it.  Softmax warpgroup
// g (query columns 32g..32g+31) writes its bf16 P^T over S columns
// [32g, 32g+16) and its dS^T over dP columns [32g, 32g+16) -- only columns
// it has read itself, so the warpgroups never wait on each other.  tcgen05
// MMAs of a CTA run in issue order, so S^T of tile n + 1 may overwrite the
// S columns once dV has been issued, and dQ may overwrite the dP columns
// once dK has been issued.  The softmax warps are software-pipelined: dS of
// tile n, then P^T of tile n + 1 (while dK and dQ of tile n run), then the
// dQ drain of tile n -- the warp of lane quarter q, warpgroup g copies
// queries 32q..32q+31, d columns [g D/4, (g+1) D/4) out of TMEM, releases the
// columns for the next dP^T, and writes the scaled fp32 values as 128-byte
// swizzled boxes of 32 columns x 64 rows.  At D = 128, dS itself was written
// into the tile's dO buffer once dV had read it; rows 0-63 of dQ go there
// after the dQ MMA has read dS, rows 64-127 into a staging buffer of their
// own.  One thread adds both halves to the fp32 dQ accumulator in global
// memory with TMA bulk reduce-adds (the SM drains reductions at ~25 B/clk,
// sharing its memory port with the tile loads), hands the dO buffer back to
// the producer as soon as the first half has been read, and frees the
// staging buffer after the second; Q goes back as soon as dK has read it.
// (At D = 64 dO is too small for dS: dS keeps a buffer of its own and both
// dQ halves go to the staging buffer.)
//
// CTA layout (640 threads, five warpgroups):
//   WG0    warp 0 TMA producer (K, V once; Q, dO, LSE2, D tiles in ring
//          order), warp 1 TMEM allocator and MMA issuer (converged; elect.sync
//          picks the issuing lane), warp 2 dQ reducer (TMA reduce-add of the
//          staged dQ halves), warp 3 idle.
//   WG1-4  P^T / dS^T / dQ drain for query columns 32(g-1)..32(g-1)+31
//          (thread = key row for P and dS, = query row for dQ); epilogue:
//          WG1-2 write dV, WG3-4 write dK (each half of the d columns).
#pragma once

#include <cstring>

#include "layout.cuh"
#include "sm103_ptx.cuh"
#include "small_kernels.cuh"
#include "profile.cuh"
#include "trace.cuh"

namespace ra {
namespace bwd {

constexpr int kBK = 128;        // keys per CTA
constexpr int kBQ = 128;        // queries per streamed tile
constexpr int kThreads = 640;
constexpr int kSoftmaxThreads = 512;   // WG1-WG4

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = 64 * 128 * 2;          // 16 KB: 128 rows x 64 bf16
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kStages = 2;                       // Q / dO / row stages
    static constexpr int kRowBytes = kBQ * 4;               // one LSE2 or D row tile
    // D = 128: dS (128 x 128 bf16, as large as a dO tile) is written into the
    // tile's dO buffer once dV has read it, so the 32 KB a separate dS buffer
    // would take hold the dQ staging of rows 64-127 instead.  D = 64: dO is
    // half that size, so dS keeps its own buffer and the staging buffer
    // holds the whole dQ tile (128 rows x 64 columns fp32).
    static constexpr bool kDsInDo = (D == 128);
    static constexpr int kStgBytes = 32768;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;
    static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
    static constexpr int kOffStg = kOffDO + kStages * kTileBytes;       // dQ staging
    static constexpr int kOffDS = kOffStg + kStgBytes;                  // dS (D = 64 only)
    static constexpr int kOffRow = kOffDS + (kDsInDo ? 0 : 2 * kBoxBytes);   // [stage][lse2 | D]
    static constexpr int kOffBar = kOffRow + kStages * 2 * kRowBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = kOffBar + kBarBytes;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColDP = 128;
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 256 + D;
};

struct BwdParams {
    const float* lse2;      // [B*H, S] LSE * log2(e)   (read directly when rows are not TMA-able)
    const float* Dvec;      // [B*H, S]
    float* dq_acc;          // [B*H*S, D] fp32, pre-zeroed
    __nv_bfloat16* dk;      // [B, H_kv, S, D] rows placed by dk_l
    __nv_bfloat16* dv;      // rows placed by dv_l
    RowLayout8 dk_l, dv_l;
    int S, P, C, causal, tiles_per_chunk;
    int H, group;           // query heads; query heads per key/value head
    float scale, scale_log2;
    int rank4;              // bit set: the q (1), k (2), v (4), dO (8) map is 4-D
    uint32_t* status;
    uint64_t wait_limit_ns;
};

// Kernel parameters (seven tensor maps and BwdParams) are kept within
// 1 KB: measured on GB300, the same kernel with 1040 bytes of parameters
// ran about 19 % slower than with 1008, with more warps stalled on long
// scoreboard dependencies.
static_assert(7 * sizeof(CUtensorMap) + sizeof(BwdParams) <= 1024, "bwd kernel parameters above 1 KB");

// Query tiles met by key tile kt of chunk j, in ring order: chunks
// i = j, j+1, ... (mod P), each chunk's tiles ascending; causal keeps
// i >= j and, in chunk j, tiles from kt on.  The sequence repeats for each
// of the `group` query heads qh0, qh0 + 1, ... that share the key tile.
struct QTiles {
    int P, C, j, causal, T, kt, group, qh0, per_head;
    int i, qt, m, left;
    __device__ __forceinline__ void init(int P_, int C_, int j_, int causal_, int T_, int kt_,
                                         int group_, int qh0_)
    {
        P = P_; C = C_; j = j_; causal = causal_; T = T_; kt = kt_; group = group_; qh0 = qh0_;
        per_head = causal ? (T - kt) + (P - 1 - j) * T : P * T;
        m = 0;
        left = per_head;
        i = j;
        qt = causal ? kt : 0;
    }
    __device__ __forceinline__ int total() const { return per_head * group; }
    __device__ __forceinline__ int q_head() const { return qh0 + m; }
    __device__ __forceinline__ int q_start() const { return i * C + qt * kBQ; }
    __device__ __forceinline__ int chunk_end() const { return (i + 1) * C; }
    __device__ __forceinline__ void next()
    {
        if (--left == 0) {               // this head is done: the next one in the group
            ++m;
            left = per_head;
            i = j;
            qt = causal ? kt : 0;
            return;
        }
        if (++qt < T) return;
        qt = 0;
        i = (i + 1 == P) ? 0 : i + 1;    // the chunk that meets j one ring step later
    }
};

// kRowTma: the per-query LSE2 / D rows arrive by TMA with the Q / dO tile
// (needs C % 4 == 0 for 16-byte aligned boxes); otherwise the softmax
// threads read them from global memory.
// kStrided: the caller's tensors use general row layouts (tensor maps may be
// 4-D, dK / dV rows are placed by p.dk_l / p.dv_l); otherwise every tensor
// is contiguous [B, heads, S, D] and the maps are 3-D over B * heads.  The
// two are separate instantiations because this kernel's speed proved
// sensitive to small changes in its generated code.
template <int D, bool kRowTma, bool kStrided>
__global__ void __launch_bounds__(kThreads, 1)
ring_bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                const __grid_constant__ CUtensorMap map_lse2, const __grid_constant__ CUtensorMap map_dvec,
                const __grid_constant__ CUtensorMap map_dq, const BwdParams p)
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
    const uint32_t sStg = base + CF::kOffStg;
    // dS of a tile in stage s: the stage's dO buffer, or the dS buffer
    auto ds_off = [&](int s) { return CF::kDsInDo ? CF::kOffDO + s * CF::kTileBytes : CF::kOffDS; };
    const uint32_t sRow = base + CF::kOffRow;
    const uint32_t bar0 = base + CF::kOffBar;
    const uint32_t bar_kv = bar0;
    // Q (with the LSE2 rows) and dO (with the D rows) of a stage arrive and
    // are released separately: Q is free once dK has read it (k_done), dO
    // once the tile is past its dS phase and, at D = 128, the dQ rows staged
    // there after dS have been reduced (do_empty, from the reducer).  The next tile's S^T can then start
    // while its dO is still loading behind the reductions that share the
    // SM's memory port.
    auto bar_q_full = [&](int s) { return bar0 + 8u * (1 + s); };
    // dO arrives and is released box by box (64 d columns each): at D = 128
    // the dQ rows staged in its first half of columns are reduced first, so
    // the next dO's first box can load, and dP^T's first k-steps run, while
    // the rest is still being read.  The D rows ride with box 1.
    auto bar_do_full = [&](int s, int x) { return bar0 + 8u * (x == 0 ? 3 + s : 27 + s); };
    auto bar_do_empty = [&](int s, int x) { return bar0 + 8u * (x == 0 ? 19 + s : 29 + s); };
    const uint32_t bar_s_full = bar0 + 8u * 5;
    const uint32_t bar_dp_full = bar0 + 8u * 6;
    const uint32_t bar_p_ready = bar0 + 8u * 7;
    const uint32_t bar_ds_ready = bar0 + 8u * 8;
    const uint32_t bar_dq_full = bar0 + 8u * 9;
    const uint32_t bar_dq_free = bar0 + 8u * 10;
    const uint32_t bar_kv_final = bar0 + 8u * 11;
    const uint32_t bar_drain = bar0 + 8u * 12;
    // dK of the stage's tile done (its Q has been read): one per stage, since
    // the MMA can finish the next tile's dK before the reducer frees this
    // stage, but not the tile after (it needs this stage back).
    auto bar_k_done = [&](int s) { return bar0 + 8u * (s == 0 ? 13u : 17u); };
    // The dQ tile is staged in two halves.  D = 128: rows 0-63 in the tile's
    // dO buffer, where dS was (free once the dQ MMA has read it), rows 64-127
    // in the staging buffer; the stage is handed back once dK has read Q and
    // the first half has been reduced.  D = 64: both halves in the staging
    // buffer; the stage is handed back once dK has read Q.
    // rows 0-63 staged by warpgroup g (d columns [g D/4, (g+1) D/4))
    auto bar_dqa_staged = [&](int g) { return bar0 + 8u * (g == 0 ? 14u : g == 1 ? 22u : g == 2 ? 23u : 26u); };
    const uint32_t bar_dqb_staged = bar0 + 8u * 15;  // rows 64-127 staged
    const uint32_t bar_stg_free = bar0 + 8u * 16;    // the staging buffer's rows have been read
    // dV of the stage's tile has read its dO (D = 128: dS may go there).
    auto bar_dv_done = [&](int s) { return bar0 + 8u * (s == 0 ? 18u : 21u); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + CF::kOffBar + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + CF::kOffBar + 200);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wg = warp >> 2;

    // ---- work item: (b*H_kv + key/value head, KV chunk j, key tile kt),
    // heaviest first ----
    const int T = p.tiles_per_chunk;
    const int items_per_head = p.P * T;
    const int bkv = blockIdx.x / items_per_head;
    const int H_kv = p.H / p.group;
    const int qh0 = (bkv / H_kv) * p.H + (bkv % H_kv) * p.group;   // first query head of the group (flat b*H + h)
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
            mbar_init(bar_q_full(s), 1);
            for (int x = 0; x < 2; ++x) {
                mbar_init(bar_do_full(s, x), 1);
                mbar_init(bar_do_empty(s, x), 1);
            }
            mbar_init(bar_dv_done(s), 1);
        }
        mbar_init(bar_s_full, 1);
        mbar_init(bar_dp_full, 1);
        mbar_init(bar_p_ready, kSoftmaxThreads);
        mbar_init(bar_ds_ready, kSoftmaxThreads);
        mbar_init(bar_dq_full, 1);
        mbar_init(bar_dq_free, kSoftmaxThreads);
        mbar_init(bar_kv_final, 1);
        mbar_init(bar_drain, 1);
        for (int s = 0; s < CF::kStages; ++s) mbar_init(bar_k_done(s), 1);
        for (int g = 0; g < 4; ++g) mbar_init(bar_dqa_staged(g), kSoftmaxThreads / 8);
        mbar_init(bar_dqb_staged, kSoftmaxThreads / 2);
        mbar_init(bar_stg_free, 1);
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
    qi.init(p.P, p.C, chunk_j, p.causal, T, kt, p.group, qh0);
    const int NT = qi.total();

    if (wg == 0) {
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------------- TMA
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            tma_prefetch_desc(&map_do);
            if constexpr (kRowTma) {
                tma_prefetch_desc(&map_lse2);
                tma_prefetch_desc(&map_dvec);
            }
            mbar_arrive_expect_tx(bar_kv, 2 * CF::kTileBytes);
            for (int x = 0; x < CF::kBoxes; ++x) {
                if constexpr (kStrided) {
                    const int b_idx = bkv / H_kv;
                    tma_load_rows(sK + x * CF::kBoxBytes, &map_k, bar_kv, 64 * x, k0, bkv - b_idx * H_kv, b_idx,
                                  H_kv, (p.rank4 & 2) != 0);
                    tma_load_rows(sV + x * CF::kBoxBytes, &map_v, bar_kv, 64 * x, k0, bkv - b_idx * H_kv, b_idx,
                                  H_kv, (p.rank4 & 4) != 0);
                } else {
                    tma_load_3d(sK + x * CF::kBoxBytes, &map_k, bar_kv, 64 * x, k0, bkv);
                    tma_load_3d(sV + x * CF::kBoxBytes, &map_v, bar_kv, 64 * x, k0, bkv);
                }
            }
            int issued_q[CF::kStages], issued_do[CF::kStages][2];
            for (int s = 0; s < CF::kStages; ++s) issued_q[s] = issued_do[s][0] = issued_do[s][1] = -1;
            bool ok = true;
            constexpr uint32_t kHalfTx = CF::kTileBytes + (kRowTma ? CF::kRowBytes : 0);
            int* tr = trace_slot(p.P);   // NULL unless the visit order is being recorded
            int visits = 0, cur_i = -1;
            for (int n = 0; n < NT; ++n, qi.next()) {
                const int s = n % CF::kStages;
                const uint32_t ph = (uint32_t)(n / CF::kStages) & 1u;
                ok = mbar_wait_poll(bar_k_done(s), ph ^ 1u, wc);   // dK of the stage's last tile read its Q
                if (!ok) break;
                const int q0 = qi.q_start();
                const int qh = qi.q_head();
                if (tr && qi.m == 0) {   // first query head of the group: record each chunk entered
                    if (qi.i != cur_i && visits < p.P) {
                        cur_i = qi.i;
                        ++visits;
                        trace_put(tr + visits * kTraceInts, qi.i, (qi.i - chunk_j + p.P) % p.P,
                                  qi.i == chunk_j ? 0 : 1, 0, q0, q0);
                    }
                    tr[visits * kTraceInts + 3] += 1;
                    tr[visits * kTraceInts + 5] = q0;
                }
                const int b_idx = qh / p.H;
                mbar_arrive_expect_tx(bar_q_full(s), kHalfTx);
                for (int x = 0; x < CF::kBoxes; ++x) {
                    if constexpr (kStrided)
                        tma_load_rows(sQ + s * CF::kTileBytes + x * CF::kBoxBytes, &map_q, bar_q_full(s),
                                      64 * x, q0, qh - b_idx * p.H, b_idx, p.H, (p.rank4 & 1) != 0);
                    else
                        tma_load_3d(sQ + s * CF::kTileBytes + x * CF::kBoxBytes, &map_q, bar_q_full(s), 64 * x, q0, qh);
                }
                if constexpr (kRowTma) tma_load_2d(sRow + s * 2 * CF::kRowBytes, &map_lse2, bar_q_full(s), q0, qh);
                issued_q[s] = (int)ph;
                // dO and the D rows, box by box: once the stage's last tile is
                // past its dS phase and (D = 128) the dQ rows staged in that
                // box have been reduced
                for (int x = 0; x < 2 && ok; ++x) {
                    ok = mbar_wait_poll(bar_do_empty(s, x), ph ^ 1u, wc);
                    if (!ok) break;
                    const bool has_box = x < CF::kBoxes;
                    const uint32_t tx = (has_box ? CF::kBoxBytes : 0) + ((x == 1 && kRowTma) ? CF::kRowBytes : 0);
                    if (tx) mbar_arrive_expect_tx(bar_do_full(s, x), tx);
                    else mbar_arrive(bar_do_full(s, x));
                    if (has_box) {
                        if constexpr (kStrided)
                            tma_load_rows(sDO + s * CF::kTileBytes + x * CF::kBoxBytes, &map_do, bar_do_full(s, x),
                                          64 * x, q0, qh - b_idx * p.H, b_idx, p.H, (p.rank4 & 8) != 0);
                        else
                            tma_load_3d(sDO + s * CF::kTileBytes + x * CF::kBoxBytes, &map_do, bar_do_full(s, x), 64 * x,
                                        q0, qh);
                    }
                    if (kRowTma && x == 1)
                        tma_load_2d(sRow + s * 2 * CF::kRowBytes + CF::kRowBytes, &map_dvec, bar_do_full(s, 1), q0, qh);
                    issued_do[s][x] = (int)ph;
                }
                if (!ok) break;
            }
            if (tr) trace_put(tr, bkv, chunk_j, kt, visits, NT, p.group);
            if (!ok) {
                WaitCtl drain{abort_flag, p.status, 200000000ull};
                volatile int dummy = 0;
                drain.abort_flag = &dummy;
                mbar_wait(bar_kv, 0, drain);
                for (int s = 0; s < CF::kStages; ++s) {
                    if (issued_q[s] >= 0) mbar_wait(bar_q_full(s), (uint32_t)issued_q[s], drain);
                    for (int x = 0; x < 2; ++x)
                        if (issued_do[s][x] >= 0) mbar_wait(bar_do_full(s, x), (uint32_t)issued_do[s][x], drain);
                }
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- MMA
            // The whole warp runs the loop converged and waits together; one
            // elected lane issues each group of MMAs and the commits, which
            // keeps the code between tcgen05.mma instructions short (the SM
            // takes one about every 48 cycles).
            constexpr uint32_t idesc_kq = idesc_bf16_f32(kBK, kBQ, false, false);   // S^T, dP^T
            constexpr uint32_t idesc_kd = idesc_bf16_f32(kBK, D, false, true);      // dV, dK
            constexpr uint32_t idesc_qd = idesc_bf16_f32(kBQ, D, true, true);       // dQ tile
            // A k-step moves a descriptor's start address (its low field,
            // address / 16) by a constant.
            // C = A(smem, K-major) * B(smem, K-major)^T over the head dim.
            auto mma_kmajor = [&](uint32_t d_tmem, uint32_t sa, uint32_t sb, int kk0 = 0, int kk1 = D / 16) {
                const uint64_t da = sdesc_sw128(sa, 16, 1024);
                const uint64_t db = sdesc_sw128(sb, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = kk0; kk < kk1; ++kk) {
                        const uint32_t off16 = ((kk >> 2) * CF::kBoxBytes + (kk & 3) * 32) >> 4;
                        mma_bf16_ss(d_tmem, da + off16, db + off16, idesc_kq, kk > 0 ? 1u : 0u);
                    }
                }
                __syncwarp();
            };
            // C += A(TMEM bf16: queries 32g..32g+31 at columns a_tmem + 32g,
            // 16 columns each) * B(smem, queries x D, MN-major).
            auto mma_ts = [&](uint32_t d_tmem, uint32_t a_tmem, uint32_t sb, bool first) {
                const uint64_t db = sdesc_sw128(sb, CF::kBoxBytes, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBQ / 16; ++kk)
                        mma_bf16_ts(d_tmem, a_tmem + (kk >> 1) * 32u + 8u * (kk & 1), db + (uint32_t)kk * (2048 >> 4),
                                    idesc_kd, (first && kk == 0) ? 0u : 1u);
                }
                __syncwarp();
            };
            // elect.sync picks the lowest lane every time, so each commit comes
            // from the thread that issued the MMAs it tracks.
            auto commit = [&](uint32_t bar) {
                if (elect_one()) mma_commit(bar);
                __syncwarp();
            };
            auto wait_all = [&](uint32_t bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
            };
            const uint64_t dk0 = sdesc_sw128(sK, CF::kBoxBytes, 1024);
            bool ok = wait_all(bar_kv, 0);
            auto issue_dq = [&](int s, uint32_t d_col) {
                // dQ tile = dS K.  A is dS^T stored [key][query] (queries
                // contiguous, MN-major); B is the K tile (d contiguous).
                const uint64_t dds0 = sdesc_sw128(base + ds_off(s), CF::kBoxBytes, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_ss(tmem + d_col, dds0 + (uint32_t)kk * (2048 >> 4), dk0 + (uint32_t)kk * (2048 >> 4),
                                    idesc_qd, kk > 0 ? 1u : 0u);
                }
                __syncwarp();
            };
            // S^T of tile n + 1 is issued right after dV of tile n (which
            // consumes the P^T in those columns), so the softmax warps can
            // start its P phase while dK and dQ of tile n run; dQ goes into
            // the dP^T columns after dK has read dS^T there.
            if (ok) ok = wait_all(bar_q_full(0), 0);
            if (ok) {
                tc_fence_after();
                mma_kmajor(tmem + CF::kColS, sK, sQ);
                commit(bar_s_full);
            }
            for (int n = 0; n < NT && ok; ++n) {
                const int s = n % CF::kStages;
                const uint32_t ph = (uint32_t)(n / CF::kStages) & 1u;
                const uint32_t par = (uint32_t)n & 1u;
                const uint32_t qs = sQ + s * CF::kTileBytes;
                const uint32_t dos = sDO + s * CF::kTileBytes;
                ok = wait_all(bar_do_full(s, 0), ph);
                if (ok && n > 0) ok = wait_all(bar_dq_free, par ^ 1u);   // dQ of tile n - 1 left the dP columns
                if (!ok) break;
                tc_fence_after();
                mma_kmajor(tmem + CF::kColDP, sV, dos, 0, 4);             // d columns 0-63 (dO box 0)
                if constexpr (CF::kBoxes == 2) {
                    ok = wait_all(bar_do_full(s, 1), ph);
                    if (!ok) break;
                    tc_fence_after();
                    mma_kmajor(tmem + CF::kColDP, sV, dos, 4, 8);         // d columns 64-127 (dO box 1)
                }
                commit(bar_dp_full);
                ok = wait_all(bar_p_ready, par);
                if (!ok) break;
                tc_fence_after();
                mma_ts(tmem + CF::kColDV, tmem + CF::kColS, dos, n == 0);
                commit(bar_dv_done(s));
                if (n + 1 < NT) {
                    const int s1 = (n + 1) % CF::kStages;
                    ok = wait_all(bar_q_full(s1), (uint32_t)((n + 1) / CF::kStages) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    mma_kmajor(tmem + CF::kColS, sK, sQ + s1 * CF::kTileBytes);
                    commit(bar_s_full);
                }
                ok = wait_all(bar_ds_ready, par);
                if (!ok) break;
                tc_fence_after();
                mma_ts(tmem + CF::kColDK, tmem + CF::kColDP, qs, n == 0);
                commit(bar_k_done(s));
                issue_dq(s, CF::kColDP);
                commit(bar_dq_full);
            }
            if (ok) commit(bar_kv_final);
            commit(bar_drain);
            WaitCtl drain{abort_flag, p.status, 200000000ull};
            volatile int dummy = 0;
            drain.abort_flag = &dummy;
            __all_sync(0xffffffffu, mbar_wait(bar_drain, 0, drain));
        } else if (warp == 2 && lane == 0) {
            // ---------------------------------------------------- dQ reducer
            // For each tile: add rows 0-63, then rows 64-127 (D / 32 boxes
            // [64 rows x 32 columns] each) to the fp32 accumulator; hand the
            // stage back once dK has read its Q and (D = 128) the first half,
            // staged in its dO buffer, has been read; then free the staging
            // buffer.  Rows past S are skipped by the TMA; rows past the chunk
            // end hold exact zeros (their P is masked to 0).
            tma_prefetch_desc(&map_dq);
            for (int n = 0; n < NT; ++n, qi.next()) {
                const int s = n % CF::kStages;
                const uint32_t par = (uint32_t)n & 1u;
                const int q0 = qi.q_start();
                const uint32_t src_a = CF::kDsInDo ? sDO + s * CF::kTileBytes : sStg;
                const uint32_t src_b = CF::kDsInDo ? sStg : sStg + CF::kStgBytes / 2;
                bool okr = true;
                if constexpr (CF::kDsInDo) {
                    // rows 0-63, box by box as each warpgroup has staged its
                    // columns; boxes 0-1 lie in dO box 0, boxes 2-3 in dO box 1
                    for (int b = 0; b < 4 && okr; ++b) {
                        okr = mbar_wait_poll(bar_dqa_staged(b), par, wc);
                        if (!okr) break;
                        tma_reduce_add_3d(&map_dq, src_a + (uint32_t)b * 8192u, 32 * b, q0, qi.q_head());
                        bulk_commit_group();
                    }
                    if (!okr) break;
                    bulk_wait_read_n<2>();              // dQ boxes 0-1 read: dO box 0 may be reloaded
                    mbar_arrive(bar_do_empty(s, 0));
                } else {
                    for (int g = 0; g < 4 && okr; ++g) okr = mbar_wait_poll(bar_dqa_staged(g), par, wc);
                    if (!okr) break;
                    // D = 64: staging began after dq_full, so every softmax
                    // warp is past its dS phase (D rows read) and dV has read dO
                    mbar_arrive(bar_do_empty(s, 0));
                    mbar_arrive(bar_do_empty(s, 1));
#pragma unroll
                    for (int b = 0; b < D / 32; ++b)
                        tma_reduce_add_3d(&map_dq, src_a + (uint32_t)b * 8192u, 32 * b, q0, qi.q_head());
                    bulk_commit_group();
                }
                if (!mbar_wait_poll(bar_dqb_staged, par, wc)) break;
#pragma unroll
                for (int b = 0; b < D / 32; ++b)
                    tma_reduce_add_3d(&map_dq, src_b + (uint32_t)b * 8192u, 32 * b, q0 + 64, qi.q_head());
                bulk_commit_group();
                if constexpr (CF::kDsInDo) {
                    bulk_wait_read_1();                  // dQ boxes 2-3 read: dO box 1 may be reloaded
                    mbar_arrive(bar_do_empty(s, 1));
                }
                bulk_wait_read_all();
                mbar_arrive(bar_stg_free);
            }
            bulk_wait_all();
        }
    } else {
        // -------------------- P^T, dS^T, dQ drain; epilogue dV / dK
        const int g = wg - 1;                            // query columns [32 g, 32 g + 32)
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int kr = (int)quarter * 32 + lane;         // key row (P, dS) / query row (dQ)
        const int kpos = k0 + kr;
        const bool key_ok = kpos < k_end;
        const uint32_t tS = tmem_addr(tmem, quarter * 32, CF::kColS + 32u * g);
        const uint32_t tDP = tmem_addr(tmem, quarter * 32, CF::kColDP + 32u * g);
        constexpr int kDqCols = D / 4;                   // dQ columns this warp drains
        const uint32_t tQ = tmem_addr(tmem, quarter * 32, CF::kColDP + (uint32_t)(kDqCols * g));
        const float sl2 = p.scale_log2;
        const float sc = p.scale;
        bool ok = true;
        // What the three phases need to know about one query tile.
        struct TileInfo {
            int n, s;
            uint32_t sph;             // phase of the stage's barriers
            int qcol0, q_valid;       // this group's first query; columns < q_valid are real
            bool diag, plain;
            size_t grow;              // row offset of the tile's head in LSE2 / D
        };
        auto info_of = [&](const QTiles& q, int n) {
            TileInfo t;
            t.n = n;
            t.s = n % CF::kStages;
            t.sph = (uint32_t)(n / CF::kStages) & 1u;
            t.qcol0 = q.q_start() + 32 * g;
            t.q_valid = q.chunk_end() - t.qcol0;
            t.diag = p.causal && q.i == chunk_j && q.qt == kt;
            t.plain = key_ok && !t.diag && t.q_valid >= 32;
            t.grow = (size_t)q.q_head() * p.S;
            return t;
        };
        auto lse_row = [&](const TileInfo& t) {
            return reinterpret_cast<const float*>(smem + CF::kOffRow + t.s * 2 * CF::kRowBytes) + 32 * g;
        };
        float pv[32];   // P^T of the tile between its P phase and its dS phase

        // P^T = exp2(S^T scale log2 e - LSE2), bf16 into the S columns.
        auto p_phase = [&](const TileInfo& t) -> bool {
            if constexpr (kRowTma) {
                // the LSE2 rows arrived with the Q tile of this stage
                if (!__all_sync(0xffffffffu, mbar_wait(bar_q_full(t.s), t.sph, wc))) return false;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(bar_s_full, (uint32_t)t.n & 1u, wc))) return false;
            tc_fence_after();
            const float* lse_s = lse_row(t);
            {
                uint32_t sv[32];
                tmem_ld32(tS, sv);
                tmem_ld_wait(sv);
                if (t.plain) {
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        float4 l4;
                        if constexpr (kRowTma) {
                            l4 = reinterpret_cast<const float4*>(lse_s)[c4];
                        } else {
                            const float* gp = p.lse2 + t.grow + t.qcol0 + 4 * c4;
                            l4 = make_float4(gp[0], gp[1], gp[2], gp[3]);
                        }
                        pv[4 * c4 + 0] = ex2_approx(fmaf(__uint_as_float(sv[4 * c4 + 0]), sl2, -l4.x));
                        pv[4 * c4 + 1] = ex2_approx(fmaf(__uint_as_float(sv[4 * c4 + 1]), sl2, -l4.y));
                        pv[4 * c4 + 2] = ex2_approx(fmaf(__uint_as_float(sv[4 * c4 + 2]), sl2, -l4.z));
                        pv[4 * c4 + 3] = ex2_approx(fmaf(__uint_as_float(sv[4 * c4 + 3]), sl2, -l4.w));
                    }
                } else {
                    // masked tile: rows past the chunk, causal diagonal, or
                    // query columns past the chunk end
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const bool valid = key_ok && c < t.q_valid && !(t.diag && t.qcol0 + c < kpos);
                        float l;
                        if constexpr (kRowTma) l = lse_s[c];
                        else l = valid ? p.lse2[t.grow + t.qcol0 + c] : 0.f;
                        const float e = ex2_approx(fmaf(__uint_as_float(sv[c]), sl2, -l));
                        pv[c] = valid ? e : 0.f;
                    }
                }
            }
            {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
                tmem_st16(tS, pk);   // P^T bf16 over S columns [32 g, 32 g + 16)
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_p_ready);
            return true;
        };

        // dS = P (dP - D): bf16 into shared memory (the dQ MMA's operand) and
        // as dS^T into the dP columns (the dK MMA's operand).
        auto ds_phase = [&](const TileInfo& t) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_dp_full, (uint32_t)t.n & 1u, wc))) return false;
            if constexpr (kRowTma) {
                // the D rows arrived with the dO tile (dP^T has read it already)
                if (!__all_sync(0xffffffffu, mbar_wait(bar_do_full(t.s, 1), t.sph, wc))) return false;
            }
            tc_fence_after();
            const float* d_s = lse_row(t) + kBQ;
            uint32_t pk[16];
            {
                uint32_t dp[32];
                tmem_ld32(tDP, dp);
                tmem_ld_wait(dp);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const int x = 4 * c4;
                    float4 d4;
                    if constexpr (kRowTma) {
                        d4 = reinterpret_cast<const float4*>(d_s)[c4];
                    } else {
                        float dd[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dd[e] = (x + e < t.q_valid) ? p.Dvec[t.grow + t.qcol0 + x + e] : 0.f;
                        d4 = make_float4(dd[0], dd[1], dd[2], dd[3]);
                    }
                    pk[2 * c4] = pack_bf16x2(pv[x] * (__uint_as_float(dp[x]) - d4.x),
                                             pv[x + 1] * (__uint_as_float(dp[x + 1]) - d4.y));
                    pk[2 * c4 + 1] = pack_bf16x2(pv[x + 2] * (__uint_as_float(dp[x + 2]) - d4.z),
                                                 pv[x + 3] * (__uint_as_float(dp[x + 3]) - d4.w));
                }
            }
            // dS to shared memory as [key][query] rows, 128-byte swizzle: the
            // 16-byte chunk c of row kr sits at chunk position c ^ (kr & 7);
            // this group's 32 queries are chunks 4 (g & 1) .. +3 of atom g / 2.
            // D = 128: the buffer is this tile's dO, once dV has read it.
            // D = 64: the dS buffer, last read by the previous tile's dQ MMA,
            // which finished before its dq_full.
            if constexpr (CF::kDsInDo) {
                if (!__all_sync(0xffffffffu, mbar_wait(bar_dv_done(t.s), t.sph, wc))) return false;
            }
            uint8_t* ds_row = smem + ds_off(t.s) + (g >> 1) * CF::kBoxBytes + kr * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(ds_row + (((4 * (g & 1) + c) ^ (kr & 7)) << 4)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            fence_proxy_async_smem();
            tmem_st16(tDP, pk);      // dS^T bf16 over dP columns [32 g, 32 g + 16)
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_ds_ready);
            return true;
        };

        // dQ drain: this warp's query rows, d columns [g D/4, (g+1) D/4),
        // out of TMEM and, scaled, into the staging boxes.
        auto drain_phase = [&](const TileInfo& t) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_dq_full, (uint32_t)t.n & 1u, wc))) return false;
            tc_fence_after();
            uint32_t a[kDqCols];
            if constexpr (kDqCols == 32) {
                tmem_ld32(tQ, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
                tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&a[0]));
            } else {
                tmem_ld16(tQ, *reinterpret_cast<uint32_t(*)[16]>(&a[0]));
                tmem_ld_wait16(*reinterpret_cast<uint32_t(*)[16]>(&a[0]));
            }
            tc_fence_before();
            mbar_arrive(bar_dq_free);                    // the dQ columns may be reused
            // Stage the scaled values: box b = (kDqCols g) / 32 holds d
            // columns [32 b, 32 b + 32) for 64 rows (8 KB), 128 bytes per
            // row, 16-byte chunk c of row r at chunk position c ^ (r & 7).
            // D = 128: rows 0-63 go to this tile's dO buffer, where dS was
            // (the dQ MMA has read it), rows 64-127 to the staging buffer.
            // D = 64: both halves to the staging buffer.  The staging buffer
            // is reused once the previous tile's rows there have been read;
            // every warp waits for that, so no staging barrier can run a
            // phase ahead of the reducer.
            const int b = (kDqCols * g) / 32;
            const int c_first = ((kDqCols * g) % 32) / 4;
            const bool upper = kr < 64;              // uniform over the warp
            if (t.n > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(bar_stg_free, (uint32_t)(t.n - 1) & 1u, wc))) return false;
            }
            uint8_t* box = upper ? (CF::kDsInDo ? smem + CF::kOffDO + t.s * CF::kTileBytes : smem + CF::kOffStg) +
                                       b * 8192 + kr * 128
                                 : smem + CF::kOffStg + (CF::kDsInDo ? 0 : CF::kStgBytes / 2) + b * 8192 +
                                       (kr - 64) * 128;
#pragma unroll
            for (int c = 0; c < kDqCols / 4; ++c)
                *reinterpret_cast<float4*>(box + (((c_first + c) ^ (kr & 7)) << 4)) =
                    make_float4(__uint_as_float(a[4 * c]) * sc, __uint_as_float(a[4 * c + 1]) * sc,
                                __uint_as_float(a[4 * c + 2]) * sc, __uint_as_float(a[4 * c + 3]) * sc);
            fence_proxy_async_smem();
            mbar_arrive(upper ? bar_dqa_staged(g) : bar_dqb_staged);
            return true;
        };

        // Software-pipelined: tile n's dS phase, then tile n + 1's P phase
        // (its S^T was issued right after dV of tile n), then tile n's dQ
        // drain -- the next P phase runs while dK and dQ of this tile are on
        // the tensor core.
        TileInfo cur = info_of(qi, 0);
        ok = p_phase(cur);
        for (int n = 0; n < NT && ok; ++n) {
            ok = ds_phase(cur);
            if (!ok) break;
            const bool more = n + 1 < NT;
            TileInfo nxt = cur;
            if (more) {
                qi.next();
                nxt = info_of(qi, n + 1);
                ok = p_phase(nxt);
                if (!ok) break;
            }
            ok = drain_phase(cur);
            if (!ok) break;
            cur = nxt;
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_kv_final, 0, wc));
        if (ok) {
            tc_fence_after();
            // WG1-2 write dV, WG3-4 write dK (times scale); each half of d
            const bool is_dk = g >= 2;
            const int col0 = (g & 1) * (D / 2);
            const uint32_t tAcc = tmem_addr(tmem, quarter * 32, (is_dk ? CF::kColDK : CF::kColDV) + col0);
            const float mul = is_dk ? p.scale : 1.f;
            __nv_bfloat16* out;
            if constexpr (kStrided) {
                const int b_idx = bkv / H_kv, h_kv = bkv - b_idx * H_kv, kr = key_ok ? kpos : 0;
                out = (is_dk ? p.dk : p.dv) + (is_dk ? p.dk_l.row(b_idx, h_kv, kr) : p.dv_l.row(b_idx, h_kv, kr)) + col0;
            } else {
                out = (is_dk ? p.dk : p.dv) + ((size_t)bkv * p.S + (size_t)(key_ok ? kpos : 0)) * D + col0;
            }
#pragma unroll
            for (int c4 = 0; c4 < D / 64; ++c4) {
                uint32_t acc[32];
                tmem_ld32(tAcc + 32u * c4, acc);
                tmem_ld_wait(acc);
                uint32_t o16[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    o16[c] = pack_bf16x2(__uint_as_float(acc[2 * c]) * mul, __uint_as_float(acc[2 * c + 1]) * mul);
                if (key_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(out + 32 * c4);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(o16[4 * v4], o16[4 * v4 + 1], o16[4 * v4 + 2], o16[4 * v4 + 3]);
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
    cudaError_t e = cudaSuccess;
    auto set = [&](const void* fn, int bytes) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    };
    set((const void*)ring_bwd_kernel<64, true, false>, Cfg<64>::kSmemBytes);
    set((const void*)ring_bwd_kernel<64, false, false>, Cfg<64>::kSmemBytes);
    set((const void*)ring_bwd_kernel<128, true, false>, Cfg<128>::kSmemBytes);
    set((const void*)ring_bwd_kernel<128, false, false>, Cfg<128>::kSmemBytes);
    set((const void*)ring_bwd_kernel<64, true, true>, Cfg<64>::kSmemBytes);
    set((const void*)ring_bwd_kernel<64, false, true>, Cfg<64>::kSmemBytes);
    set((const void*)ring_bwd_kernel<128, true, true>, Cfg<128>::kSmemBytes);
    set((const void*)ring_bwd_kernel<128, false, true>, Cfg<128>::kSmemBytes);
    return e;
}

struct Launch {
    const void *q, *k, *v, *o, *dO;
    const float* lse;
    void *dq, *dk, *dv;
    RowLayout lq, lk, lv, lo, ldo, ldq, ldk, ldv;   // row layouts of the caller's tensors
    int B, H, H_kv, S, d, P, causal;
    float scale;
    void* workspace;
    uint32_t* status;
    int num_sms;
    uint64_t wait_limit_ns;
    cudaStream_t stream;
    // map of a bf16 tensor with the given row layout (3-D {d, S, B * heads}
    // when batch and head fold into one index, else 4-D; *rank4 says which)
    int (*encode)(CUtensorMap*, const void*, int B, int heads, int S, int d, RowLayout, int rows, bool* rank4);
    int (*encode_rows)(CUtensorMap*, const float*, int, int);
    int (*encode_acc)(CUtensorMap*, float*, int, int, int);
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
    auto same = [](const RowLayout& a, const RowLayout& b) { return a.sb == b.sb && a.sh == b.sh && a.ss == b.ss; };
    const RowLayout cq = normalized(contiguous_layout(L.H, L.S, L.d), L.B, L.H, L.S),
                    ckv = normalized(contiguous_layout(L.H_kv, L.S, L.d), L.B, L.H_kv, L.S);
    const bool strided = !(same(L.lq, cq) && same(L.lo, cq) && same(L.ldo, cq) && same(L.ldq, cq) &&
                           same(L.lk, ckv) && same(L.lv, ckv) && same(L.ldk, ckv) && same(L.ldv, ckv));
    {
        prof::Scope ps(prof::kBwdPrep, L.stream);
        auto prep = [&](auto kern) {
            kern<<<(unsigned)blocks, 256, 0, L.stream>>>(o, L.lo, dO, L.ldo, L.lse, Dvec, lse2, (long long)rows,
                                                         L.H, L.S);
        };
        if (L.d == 128) {
            if (strided) prep(bwd_prep_kernel<128, true>); else prep(bwd_prep_kernel<128, false>);
        } else {
            if (strided) prep(bwd_prep_kernel<64, true>); else prep(bwd_prep_kernel<64, false>);
        }
        ps.done();
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = e; return -3; }

    CUtensorMap mq, mk, mv, mdo, mlse, mdv, mdq;
    const int BH = L.B * L.H;
    const int BHkv = L.B * L.H_kv;
    const int C = L.S / L.P;
    const bool row_tma = (C % 4) == 0;
    bool r4q = false, r4k = false, r4v = false, r4do = false;
    if (L.encode(&mq, L.q, L.B, L.H, L.S, L.d, L.lq, kBQ, &r4q) ||
        L.encode(&mk, L.k, L.B, L.H_kv, L.S, L.d, L.lk, kBK, &r4k) ||
        L.encode(&mv, L.v, L.B, L.H_kv, L.S, L.d, L.lv, kBK, &r4v) ||
        L.encode(&mdo, L.dO, L.B, L.H, L.S, L.d, L.ldo, kBQ, &r4do)) {
        *err = cudaErrorInvalidValue;
        return -3;
    }
    if (L.encode_acc(&mdq, dq_acc, BH, L.S, L.d)) {
        *err = cudaErrorInvalidValue;
        return -3;
    }
    std::memset(&mlse, 0, sizeof(mlse));
    std::memset(&mdv, 0, sizeof(mdv));
    if (row_tma && (L.encode_rows(&mlse, lse2, BH, L.S) || L.encode_rows(&mdv, Dvec, BH, L.S))) {
        *err = cudaErrorInvalidValue;
        return -3;
    }
    BwdParams prm;
    prm.lse2 = lse2;
    prm.Dvec = Dvec;
    prm.dq_acc = dq_acc;
    prm.dk = static_cast<__nv_bfloat16*>(L.dk);
    prm.dv = static_cast<__nv_bfloat16*>(L.dv);
    prm.dk_l = pack8(L.ldk);
    prm.dv_l = pack8(L.ldv);
    prm.rank4 = (r4q ? 1 : 0) | (r4k ? 2 : 0) | (r4v ? 4 : 0) | (r4do ? 8 : 0);
    prm.S = L.S;
    prm.P = L.P;
    prm.C = C;
    prm.causal = L.causal;
    prm.tiles_per_chunk = (prm.C + kBK - 1) / kBK;
    prm.H = L.H;
    prm.group = L.H / L.H_kv;
    prm.scale = L.scale;
    prm.scale_log2 = (float)((double)L.scale * 1.4426950408889634);
    prm.status = L.status;
    prm.wait_limit_ns = L.wait_limit_ns;
    const long long grid = (long long)BHkv * L.P * prm.tiles_per_chunk;
    {
        prof::Scope ps(prof::kBwdMain, L.stream);
        const dim3 g((unsigned)grid), b(kThreads);
        auto main_kernel = [&](auto kern, int smem) {
            kern<<<g, b, smem, L.stream>>>(mq, mk, mv, mdo, mlse, mdv, mdq, prm);
        };
        constexpr int s128 = Cfg<128>::kSmemBytes, s64 = Cfg<64>::kSmemBytes;
        if (L.d == 128) {
            if (row_tma) {
                if (strided) main_kernel(ring_bwd_kernel<128, true, true>, s128);
                else main_kernel(ring_bwd_kernel<128, true, false>, s128);
            } else {
                if (strided) main_kernel(ring_bwd_kernel<128, false, true>, s128);
                else main_kernel(ring_bwd_kernel<128, false, false>, s128);
            }
        } else {
            if (row_tma) {
                if (strided) main_kernel(ring_bwd_kernel<64, true, true>, s64);
                else main_kernel(ring_bwd_kernel<64, true, false>, s64);
            } else {
                if (strided) main_kernel(ring_bwd_kernel<64, false, true>, s64);
                else main_kernel(ring_bwd_kernel<64, false, false>, s64);
            }
        }
        ps.done();
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = e; return -3; }
    const long long n8 = (long long)(rows * L.d / 8);
    long long cb = (n8 + 255) / 256;
    if (cb > cap) cb = cap;
    {
        prof::Scope ps(prof::kDqConvert, L.stream);
        auto conv = [&](auto kern) {
            kern<<<(unsigned)cb, 256, 0, L.stream>>>(dq_acc, static_cast<__nv_bfloat16*>(L.dq), L.ldq, n8, L.H, L.S);
        };
        if (L.d == 128) {
            if (strided) conv(dq_convert_kernel<128, true>); else conv(dq_convert_kernel<128, false>);
        } else {
            if (strided) conv(dq_convert_kernel<64, true>); else conv(dq_convert_kernel<64, false>);
        }
        ps.done();
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = e; return -3; }
    return 0;
}

}  // namespace bwd
}  // namespace ra
