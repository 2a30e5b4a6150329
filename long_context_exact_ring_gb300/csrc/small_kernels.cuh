// small_kernels.cuh -- the memory-bound kernels of the library:
//   merge_partials_kernel  log-sum-exp merge of two partial attentions
//   bwd_prep_kernel        D_r = sum_k dO_rk O_rk and LSE in log2 units
//   dq_convert_kernel      fp32 dQ accumulator -> bf16 dQ
#pragma once

#include "layout.cuh"
#include "sm103_ptx.cuh"

namespace ra {

// Merge of two partial results of the same query rows ("Context
// Parallelism" guide, section 2: partial attention results merged with the
// online-softmax statistics; "Training Long-Context Models Without OOM:
// Ring Attention", "Ring Attention Demystified": running row maximum and
// sum of exponentials):
//     m = max(lse_a, lse_b),  w_a = exp(lse_a - m),  w_b = exp(lse_b - m)
//     O = (w_a O_a + w_b O_b) / (w_a + w_b),  lse = m + ln(w_a + w_b).
// (0, -inf) is the identity; two -inf rows give (0, -inf).
//
// One warp per row (four rows per warp and iteration when d is a multiple
// of 4 up to 128, so every lane has eight 16-byte loads in flight before it
// computes), grid-stride over rows.  A row's LSE pair is read by every lane
// before lane 0 writes the merged LSE, so lse_out may alias lse_a (and o_out
// may alias o_a: each element is read, then written, by the same lane).
__device__ __forceinline__ void merge_weights(float la, float lb, float& ca, float& cb, float& lse)
{
    const float m = fmaxf(la, lb);
    if (m == -INFINITY) {
        ca = 0.f; cb = 0.f; lse = -INFINITY;
        return;
    }
    const float wa = expf(la - m);
    const float wb = expf(lb - m);
    const float inv = 1.f / (wa + wb);
    ca = wa * inv;
    cb = wb * inv;
    lse = m + logf(wa + wb);
}

__global__ void __launch_bounds__(256)
merge_partials_kernel(const float* o_a, const float* lse_a, const float* __restrict__ o_b,
                      const float* lse_b, float* o_out, float* lse_out, long long rows, int d)
{
    const long long warp_global = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long warp_count = ((long long)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    if ((d & 3) == 0 && d <= 128) {
        constexpr int R = 4;
        const int nv = d >> 2;                      // float4 per row; lanes >= nv idle
        const float4* a4 = reinterpret_cast<const float4*>(o_a);
        const float4* b4 = reinterpret_cast<const float4*>(o_b);
        float4* o4 = reinterpret_cast<float4*>(o_out);
        for (long long r0 = warp_global * R; r0 < rows; r0 += warp_count * R) {
            float la[R], lb[R];
            float4 a[R], b[R];
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const long long r = r0 + k;
                la[k] = lb[k] = -INFINITY;
                a[k] = b[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < rows) {
                    la[k] = lse_a[r];
                    lb[k] = lse_b[r];
                    if (lane < nv) {
                        a[k] = a4[r * nv + lane];
                        b[k] = b4[r * nv + lane];
                    }
                }
            }
            float lo[R];
#pragma unroll
            for (int k = 0; k < R; ++k) {
                float ca, cb;
                merge_weights(la[k], lb[k], ca, cb, lo[k]);
                const long long r = r0 + k;
                if (r < rows && lane < nv)
                    o4[r * nv + lane] = make_float4(ca * a[k].x + cb * b[k].x, ca * a[k].y + cb * b[k].y,
                                                    ca * a[k].z + cb * b[k].z, ca * a[k].w + cb * b[k].w);
            }
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < R; ++k)
                    if (r0 + k < rows) lse_out[r0 + k] = lo[k];
            }
        }
        return;
    }
    for (long long r = warp_global; r < rows; r += warp_count) {
        float ca, cb, lo;
        merge_weights(lse_a[r], lse_b[r], ca, cb, lo);
        const size_t base = (size_t)r * d;
        for (int x = lane; x < d; x += 32) o_out[base + x] = ca * o_a[base + x] + cb * o_b[base + x];
        __syncwarp();
        if (lane == 0) lse_out[r] = lo;
    }
}

// Backward preparation (contiguous tensors: each lane loads 8 bf16 -- 16
// bytes -- of a row of O and of dO, D / 8 lanes per row, four rows' loads
// per lane in flight before the reductions; strided tensors: one warp per
// row):
//   D_r = sum_k dO_rk * O_rk (fp32 accumulate of the bf16 inputs) and
//   lse2_r = LSE_r * log2(e) (the exponent base the main kernel uses).
// Row r = (b H + h) S + s of D and lse2.  kStrided: O and dO rows are
// placed by their layouts; otherwise both are contiguous [B * H * S, D].
template <int D, bool kStrided>
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, RowLayout lo, const __nv_bfloat16* __restrict__ dO,
                RowLayout ldo, const float* __restrict__ lse, float* __restrict__ Dvec,
                float* __restrict__ lse2, long long rows, int H, int S)
{
    const long long warp_global = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long warp_count = ((long long)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    // Strided: each warp takes a contiguous run of rows; contiguous: warps
    // stride over rows.  Both give each lane 8 bf16 (16 bytes) of a row of O
    // and of dO, D / 8 lanes per row, and sum in the same order, so D comes
    // out bit-identical for any row layout.
    const long long per = kStrided ? (rows + warp_count - 1) / warp_count : 0;
    const long long r = kStrided ? warp_global * per : warp_global;
    const long long r_end = kStrided ? min(rows, r + per) : rows;
    if constexpr (!kStrided) {
        // lanes take 8 bf16 (16 bytes) of a row: kLpr lanes per row, kRpl
        // rows per warp-wide load, four loads per tensor in flight per lane
        constexpr int kLpr = D / 8, kRpl = 32 / kLpr, R = 4 * kRpl;
        const int g = lane / kLpr;
        const size_t c8 = (size_t)(lane % kLpr) * 8;
        for (long long r0 = warp_global * R; r0 < rows; r0 += warp_count * R) {
            uint4 a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const long long rr = min(r0 + i * kRpl + g, rows - 1);
                a[i] = *reinterpret_cast<const uint4*>(o + (size_t)rr * D + c8);
                b[i] = *reinterpret_cast<const uint4*>(dO + (size_t)rr * D + c8);
            }
            float acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[i]);
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[i]);
                float x = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 fa = __bfloat1622float2(a2[e]);
                    const float2 fb = __bfloat1622float2(b2[e]);
                    x = fmaf(fa.x, fb.x, x);
                    x = fmaf(fa.y, fb.y, x);
                }
                acc[i] = x;
            }
#pragma unroll
            for (int off = kLpr / 2; off > 0; off >>= 1)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
            if (lane % kLpr == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const long long rr = r0 + i * kRpl + g;
                    if (rr < rows) {
                        Dvec[rr] = acc[i];
                        lse2[rr] = lse[rr] * 1.4426950408889634f;
                    }
                }
            }
        }
    } else {
        constexpr int kLpr = D / 8, kRpl = 32 / kLpr;
        const int g = lane / kLpr;
        const size_t c8 = (size_t)(lane % kLpr) * 8;
        for (long long r0 = r; r0 < r_end; r0 += kRpl) {
            const long long rr = min(r0 + g, r_end - 1);
            const int bh = (int)(rr / S);   // rows < 2^31 (checked by the host)
            const int ps = (int)(rr - (long long)bh * S);
            const int bq = bh / H, hq = bh - bq * H;
            const uint4 a = *reinterpret_cast<const uint4*>(o + lo.row(bq, hq, ps) + c8);
            const uint4 b = *reinterpret_cast<const uint4*>(dO + ldo.row(bq, hq, ps) + c8);
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = __bfloat1622float2(a2[e]);
                const float2 fb = __bfloat1622float2(b2[e]);
                x = fmaf(fa.x, fb.x, x);
                x = fmaf(fa.y, fb.y, x);
            }
#pragma unroll
            for (int off = kLpr / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
            if (lane % kLpr == 0 && r0 + g < r_end) {
                Dvec[r0 + g] = x;
                lse2[r0 + g] = lse[r0 + g] * 1.4426950408889634f;
            }
        }
    }
}

// dQ (fp32 accumulator [B*H*S, D], already scaled) -> bf16, 8 elements per
// thread; kStrided: the rows are placed by `ldq`, else contiguous.
template <int D, bool kStrided>
__global__ void __launch_bounds__(256)
dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, RowLayout ldq,
                  long long n8, int H, int S)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        size_t dst = (size_t)i * 8;
        if constexpr (kStrided) {
            const int r = (int)(i / (D / 8));   // rows < 2^31 (checked by the host)
            const int col = (int)(i % (D / 8)) * 8;
            const int bh = r / S;
            dst = ldq.row(bh / H, bh % H, r - bh * S) + col;
        }
        const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
        uint4 out;
        out.x = pack_bf16x2(a.x, a.y);
        out.y = pack_bf16x2(a.z, a.w);
        out.z = pack_bf16x2(b.x, b.y);
        out.w = pack_bf16x2(b.z, b.w);
        *reinterpret_cast<uint4*>(dq + dst) = out;
    }
}

// fp32 -> bf16 with round-to-nearest-even, 8 elements per thread and
// iteration (two 16-byte loads, one 16-byte store); n8 = elements / 8.
// The fp32-input forward rounds its inputs with it before the bf16 MMAs.
__global__ void __launch_bounds__(256)
f32_to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out, long long n8)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const float4 a = reinterpret_cast<const float4*>(in)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(in)[2 * i + 1];
        uint4 o;
        o.x = pack_bf16x2(a.x, a.y);
        o.y = pack_bf16x2(a.z, a.w);
        o.z = pack_bf16x2(b.x, b.y);
        o.w = pack_bf16x2(b.z, b.w);
        reinterpret_cast<uint4*>(out)[i] = o;
    }
}

}  // namespace ra
