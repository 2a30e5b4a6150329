// layout.cuh -- where a row of a [B, H, S, d] tensor lives.
//
// Every tensor the caller passes (Q, K, V, O, dO, dQ, dK, dV) is a set of
// d-element rows indexed by (batch b, head h, position s); the d elements
// of a row are contiguous, and the rows sit at element offset
//     b * sb + h * sh + s * ss.
// The contiguous [B, H, S, d] layout is (sb, sh, ss) = (H S d, S d, d); the
// sequence-major [B, S, H, d] layout is (S H d, d, H d).  Internal buffers
// (LSE, D, the fp32 dQ accumulator, ring receive buffers) stay contiguous.
#pragma once

#include <cstddef>
#include <cstdint>

namespace ra {

struct RowLayout {
    long long sb, sh, ss;   // element strides of batch, head and position

    __host__ __device__ __forceinline__ size_t row(int b, int h, int s) const
    {
        return (size_t)((long long)b * sb + (long long)h * sh + (long long)s * ss);
    }
};

// The layout with the strides of extent-1 dimensions set to 0 (they are
// never used), so that equal placements compare equal.
__host__ __device__ inline RowLayout normalized(RowLayout l, int B, int heads, int S)
{
    if (B <= 1) l.sb = 0;
    if (heads <= 1) l.sh = 0;
    if (S <= 1) l.ss = 0;
    return l;
}

// The same layout packed into 12 bytes, for kernels whose parameter block
// must stay small: strides in units of 8 elements.  Every stride the
// library accepts is a multiple of 8 elements below 2^35, so each fits.
struct RowLayout8 {
    uint32_t sb8, sh8, ss8;

    __host__ __device__ __forceinline__ size_t row(int b, int h, int s) const
    {
        return ((size_t)b * sb8 + (size_t)h * sh8 + (size_t)s * ss8) * 8;
    }
};

__host__ __device__ inline RowLayout8 pack8(const RowLayout& l)
{
    return RowLayout8{(uint32_t)(l.sb / 8), (uint32_t)(l.sh / 8), (uint32_t)(l.ss / 8)};
}

__host__ __device__ inline RowLayout contiguous_layout(int H, int S, int d)
{
    return RowLayout{(long long)H * S * d, (long long)S * d, (long long)d};
}

}  // namespace ra
