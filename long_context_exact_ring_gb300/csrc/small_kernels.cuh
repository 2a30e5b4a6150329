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

// Backward preparation, one warp per row (contiguous tensors: four rows per
// warp and iteration, all loads issued before the reductions):
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
    constexpr int kPer = D / 32;   // elements per lane (2 or 4)
    // Strided: each warp takes a contiguous run of rows and steps (position,
    // head, batch) along it, so the only divisions are at its start.
    // Contiguous: warps stride over rows.
    const long long per = kStrided ? (rows + warp_count - 1) / warp_count : 0;
    long long r = kStrided ? warp_global * per : warp_global;
    const long long r_end = kStrided ? min(rows, r + per) : rows;
    int pos = 0, bi = 0, hi = 0;
    if constexpr (kStrided) {
        if (r >= r_end) return;
        const int bh0 = (int)r / S;          // rows < 2^31 (checked by the host)
        pos = (int)r - bh0 * S;
        bi = bh0 / H;
        hi = bh0 - bi * H;
    }
    const size_t col = (size_t)lane * kPer;
    if constexpr (!kStrided) {
        // four rows per warp and iteration: every lane has eight loads in
        // flight before the reductions
        constexpr int R = 4;
        for (long long r0 = warp_global * R; r0 < rows; r0 += warp_count * R) {
            float acc[R];
            if constexpr (kPer == 4) {
                uint2 a[R], b[R];
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    const long long rr = min(r0 + k, rows - 1);
                    a[k] = *reinterpret_cast<const uint2*>(o + (size_t)rr * D + col);
                    b[k] = *reinterpret_cast<const uint2*>(dO + (size_t)rr * D + col);
                }
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
                    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[k]);
                    float x = 0.f;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float2 fa = __bfloat1622float2(a2[e]);
                        const float2 fb = __bfloat1622float2(b2[e]);
                        x = fmaf(fa.x, fb.x, x);
                        x = fmaf(fa.y, fb.y, x);
                    }
                    acc[k] = x;
                }
            } else {
                __nv_bfloat162 a[R], b[R];
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    const long long rr = min(r0 + k, rows - 1);
                    a[k] = *reinterpret_cast<const __nv_bfloat162*>(o + (size_t)rr * D + col);
                    b[k] = *reinterpret_cast<const __nv_bfloat162*>(dO + (size_t)rr * D + col);
                }
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    const float2 fa = __bfloat1622float2(a[k]);
                    const float2 fb = __bfloat1622float2(b[k]);
                    acc[k] = fmaf(fa.y, fb.y, fa.x * fb.x);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int k = 0; k < R; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
            if (lane < R && r0 + lane < rows) {
                float x = acc[0];
#pragma unroll
                for (int k = 1; k < R; ++k) if (lane == k) x = acc[k];
                Dvec[r0 + lane] = x;
                lse2[r0 + lane] = lse[r0 + lane] * 1.4426950408889634f;
            }
        }
    } else {
    for (; r < r_end; ++r) {   // strided: each warp walks its own run of rows
        const size_t base_o = lo.row(bi, hi, pos) + col;
        const size_t base_do = ldo.row(bi, hi, pos) + col;
        if (++pos == S) {
            pos = 0;
            if (++hi == H) { hi = 0; ++bi; }
        }
        float acc = 0.f;
        if constexpr (kPer == 4) {
            const uint2 a = *reinterpret_cast<const uint2*>(o + base_o);
            const uint2 b = *reinterpret_cast<const uint2*>(dO + base_do);
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const float2 fa = __bfloat1622float2(a2[x]);
                const float2 fb = __bfloat1622float2(b2[x]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
        } else {
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(o + base_o);
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(dO + base_do);
            const float2 fa = __bfloat1622float2(a);
            const float2 fb = __bfloat1622float2(b);
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            Dvec[r] = acc;
            lse2[r] = lse[r] * 1.4426950408889634f;
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
