// ring_attn.cu -- the C-ABI boundary of libringattn.so: argument
// validation, TMA descriptor set-up, per-device state and kernel launches.
// Declarations and the contract of every entry point: include/ring_attn.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ring_attn.h"
#include "profile.cuh"
#include "fwd_kernel.cuh"
#include "bwd_kernel.cuh"
#include "small_kernels.cuh"

namespace {

// One status word per device (bit flags, see ra::kStatus*).
__device__ uint32_t g_status_word;

thread_local char g_last_error[256] = "";
std::atomic<unsigned long long> g_wait_limit_ns{4000000000ull};

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    uint32_t* status = nullptr;   // device address of g_status_word
    int num_sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int fail_cuda(cudaError_t e, const char* what)
{
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
    return RA_ERR_CUDA;
}

// Per-device set-up, once per device: resolve the status word's device
// address, raise the kernels' shared-memory limits, find the TMA encoder.
int device_state(DeviceState** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    DeviceState& st = g_dev[dev];
    if (st.ready) {
        *out = &st;
        return RA_OK;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!st.ready) {
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail_cuda(e == cudaSuccess ? cudaErrorNotSupported : e,
                                 "cuTensorMapEncodeTiled lookup");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_status_word);
        if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(status)");
        st.status = static_cast<uint32_t*>(addr);
        e = cudaMemset(st.status, 0, sizeof(uint32_t));
        if (e != cudaSuccess) return fail_cuda(e, "cudaMemset(status)");
        e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
        e = cudaFuncSetAttribute(ra::fwd::ring_fwd_kernel<64>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 ra::fwd::Cfg<64>::kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ra::fwd::ring_fwd_kernel<128>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     ra::fwd::Cfg<128>::kSmemBytes);
        if (e == cudaSuccess) e = ra::bwd::configure_kernels();
        if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute");
        st.ready = true;
    }
    *out = &st;
    return RA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tiled map over a bf16 tensor of d-element rows placed by `lay`: box of 64
// columns x `rows` rows of one (batch, head), 128-byte swizzle, rows past S
// read as zero.  When batch and head fold into one index with a single
// stride (B == 1, one head, or sb == heads * sh) the map is 3-D
// {d, S, B * heads}; otherwise it is 4-D {d, S, heads, B}.  *rank4 says
// which.  A dimension of extent 1 is never stepped along, so an invalid
// stride there is replaced by a valid placeholder.
int make_map(CUtensorMap* map, const void* ptr, int B, int heads, int S, int d, ra::RowLayout lay,
             int rows, bool* rank4)
{
    auto stride = [&](long long st, int extent) { return (cuuint64_t)((extent > 1 ? st : d) * 2); };
    long long bh_stride = 0;
    bool fold = true;
    if (B == 1) bh_stride = lay.sh;
    else if (heads == 1) bh_stride = lay.sb;
    else if (lay.sb == (long long)heads * lay.sh) bh_stride = lay.sh;
    else fold = false;
    CUresult r;
    if (fold) {
        const int BH = B * heads;
        cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)BH};
        cuuint64_t strides[2] = {stride(lay.ss, S), stride(bh_stride, BH)};
        cuuint32_t box[3] = {64u, (cuuint32_t)rows, 1u};
        cuuint32_t estr[3] = {1u, 1u, 1u};
        r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)heads, (cuuint64_t)B};
        cuuint64_t strides[3] = {stride(lay.ss, S), stride(lay.sh, heads), stride(lay.sb, B)};
        cuuint32_t box[4] = {64u, (cuuint32_t)rows, 1u, 1u};
        cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
        r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed (%d)",
                      (int)r);
        return RA_ERR_CUDA;
    }
    *rank4 = !fold;
    return RA_OK;
}

// A caller's row layout is usable when every dimension of extent > 1 has a
// positive stride that is a multiple of 8 elements (16 bytes, as the tensor
// maps and the 16-byte row stores need) and below 2^35 elements (so that
// stride / 8 fits in 32 bits).  A stride of an extent-1 dimension is never
// used; it is zeroed so the packed form stays exact.
bool layout_ok(ra::RowLayout& l, int B, int heads, int S)
{
    auto ok = [](long long st, int extent) {
        return extent <= 1 || (st > 0 && st % 8 == 0 && st < (1ll << 35));
    };
    if (!(ok(l.sb, B) && ok(l.sh, heads) && ok(l.ss, S))) return false;
    l = ra::normalized(l, B, heads, S);
    return true;
}

// Layout from a caller's stride triple (batch, head, position), or the
// contiguous [B, heads, S, d] layout when the pointer is NULL.
ra::RowLayout layout_from(const long long* strides, int heads, int S, int d)
{
    if (!strides) return ra::contiguous_layout(heads, S, d);
    return ra::RowLayout{strides[0], strides[1], strides[2]};
}

// 2-D map over a [B*H, S] fp32 row vector: boxes of 128 consecutive rows of
// one head, no swizzle.  Needs S % 4 == 0 (16-byte row stride).
int make_row_map(CUtensorMap* map, const float* ptr, int BH, int S)
{
    cuuint64_t dims[2] = {(cuuint64_t)S, (cuuint64_t)BH};
    cuuint64_t strides[1] = {(cuuint64_t)S * 4};
    cuuint32_t box[2] = {128u, 1u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled (rows) failed (%d)",
                      (int)r);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

// 3-D map over the fp32 dQ accumulator [B*H, S, d]: boxes of 32 columns x
// 64 rows x 1 head with 128-byte swizzle, used for TMA reduce-adds (a
// 128-row dQ tile is staged and added in two halves).  Rows past S are not
// written.
int make_acc_map(CUtensorMap* map, float* ptr, int BH, int S, int d)
{
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)S * d * 4};
    cuuint32_t box[3] = {32u, 64u, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled (dQ) failed (%d)",
                      (int)r);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}

// Shape checks shared by the forward and backward passes.
int check_shape(int B, int H, int S, int d, int P, int causal, float scale)
{
    if (B < 0 || H < 0 || S < 0 || P < 1) return RA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return RA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return RA_ERR_INVALID_ARG;
    if (S % P != 0) return RA_ERR_INVALID_ARG;   // equal contiguous chunks only
    if (d != 64 && d != 128) return RA_ERR_UNSUPPORTED;
    if ((long long)B * H > (1ll << 30)) return RA_ERR_UNSUPPORTED;
    if ((long long)B * H * S >= (1ll << 31)) return RA_ERR_UNSUPPORTED;   // row indices are 32-bit
    return RA_OK;
}

// Scratch of ring_attn_bwd_noalloc, for callers that cannot allocate:
// the backward workspace (fp32 dQ accumulator, D and LSE2 rows) in static
// device memory, one copy per device that loads the library.  Host code
// must not pass the symbol itself to a kernel (on the host it names a
// stand-in, not the device array); it uses the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RING_ATTN_NOALLOC_SCRATCH_BYTES];

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.
int noalloc_scratch(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(noalloc scratch)");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return RA_OK;
}

}  // namespace

extern "C" {

const char* ring_attn_status_string(int status)
{
    switch (status) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_DEVICE_TIMEOUT: return "RA_ERR_DEVICE_TIMEOUT";
    default: return "RA_UNKNOWN_STATUS";
    }
}

const char* ring_attn_last_error(void) { return g_last_error; }

int ring_attn_set_wait_limit_ns(unsigned long long ns)
{
    g_wait_limit_ns.store(ns == 0 ? 4000000000ull : ns);
    return RA_OK;
}

int ring_attn_schedule(int P, int causal, int i, int* out_j, int* out_kind, int cap)
{
    if (P < 1 || i < 0 || i >= P || (causal != 0 && causal != 1) || cap < 0)
        return RA_ERR_INVALID_ARG;
    const int count = causal ? i + 1 : P;
    if (cap == 0 && !out_j && !out_kind) return count;
    if (!out_j || !out_kind || cap < count) return RA_ERR_INVALID_ARG;
    int n = 0;
    for (int t = 0; t < P; ++t) {
        const int j = ((i - t) % P + P) % P;
        if (causal && j > i) continue;
        out_j[n] = j;
        out_kind[n] = (j == i) ? 0 : 1;
        ++n;
    }
    return n;
}

}  // extern "C"

namespace {

// o32: when set, O is written in fp32 (contiguous [B, H, S, d]) there and
// `o` is not used.
int fwd_impl(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, ra_bf16* o, float* lse, int B,
             int H, int H_kv, int S, int d, int P, int causal, float scale, void* stream,
             const long long* qs = nullptr, const long long* ks = nullptr,
             const long long* vs = nullptr, const long long* os = nullptr, float* o32 = nullptr)
{
    int rc = check_shape(B, H, S, d, P, causal, scale);
    if (rc != RA_OK) return rc;
    if (H_kv < 1 ? H != 0 : (H % H_kv) != 0) return RA_ERR_INVALID_ARG;
    if ((long long)B * H * S == 0) return RA_OK;   // empty: nothing to launch or read
    ra::RowLayout lq = layout_from(qs, H, S, d), lk = layout_from(ks, H_kv, S, d),
                  lv = layout_from(vs, H_kv, S, d), lo = layout_from(os, H, S, d);
    if (!layout_ok(lq, B, H, S) || !layout_ok(lk, B, H_kv, S) || !layout_ok(lv, B, H_kv, S) ||
        !layout_ok(lo, B, H, S))
        return RA_ERR_INVALID_ARG;
    if ((long long)B * H * S == 0) return RA_OK;
    if (o32) o = reinterpret_cast<ra_bf16*>(o32);   // only checked below, never written as bf16
    if (!q || !k || !v || !o || !lse) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return RA_ERR_INVALID_ARG;
    const int C = S / P;
    const long long pairs = (C + ra::fwd::kRowsPerCta - 1) / ra::fwd::kRowsPerCta;
    const long long grid = (long long)B * H * P * pairs;
    if (grid > 0x7fffffffll) return RA_ERR_UNSUPPORTED;

    DeviceState* st = nullptr;
    rc = device_state(&st);
    if (rc != RA_OK) return rc;
    CUtensorMap mq, mk, mv;
    const int BH = B * H;
    bool r4q = false, r4k = false, r4v = false;
    if ((rc = make_map(&mq, q, B, H, S, d, lq, ra::fwd::kBM, &r4q)) != RA_OK) return rc;
    if ((rc = make_map(&mk, k, B, H_kv, S, d, lk, ra::fwd::kBN, &r4k)) != RA_OK) return rc;
    if ((rc = make_map(&mv, v, B, H_kv, S, d, lv, ra::fwd::kBN, &r4v)) != RA_OK) return rc;

    ra::fwd::FwdParams prm;
    prm.rank4 = (r4q ? 1 : 0) | (r4k ? 2 : 0) | (r4v ? 4 : 0);
    prm.o = reinterpret_cast<__nv_bfloat16*>(o);
    prm.lo = lo;
    prm.lse = lse;
    prm.S = S;
    prm.P = P;
    prm.C = C;
    prm.causal = causal;
    prm.pairs_per_chunk = (int)pairs;
    prm.H = H;
    prm.group = H / H_kv;
    prm.step = -1;
    prm.BH = BH;
    prm.o32 = o32;
    prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
    prm.status = st->status;
    prm.wait_limit_ns = g_wait_limit_ns.load();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ra::prof::Scope ps(ra::prof::kFwd, s);
    if (d == 128)
        ra::fwd::ring_fwd_kernel<128><<<(unsigned)grid, ra::fwd::kThreads,
                                        ra::fwd::Cfg<128>::kSmemBytes, s>>>(mq, mk, mv, prm);
    else
        ra::fwd::ring_fwd_kernel<64><<<(unsigned)grid, ra::fwd::kThreads,
                                       ra::fwd::Cfg<64>::kSmemBytes, s>>>(mq, mk, mv, prm);
    ps.done();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "ring_fwd_kernel launch");
    return RA_OK;
}

int bwd_impl(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, const ra_bf16* o,
             const float* lse, const ra_bf16* dO, ra_bf16* dq, ra_bf16* dk, ra_bf16* dv, int B,
             int H, int H_kv, int S, int d, int P, int causal, float scale, void* workspace,
             size_t workspace_bytes, void* stream, const long long* const* strides = nullptr);

// ---------------------------------------------------------------------------
// Emulated ring: P logical ranks on one GPU
// ---------------------------------------------------------------------------
// Per device: a non-blocking copy stream (the "interconnect") and the events
// that order it against the compute stream; created on first use, kept.
struct RingRuntime {
    bool ready = false;
    cudaStream_t copy = nullptr;
    cudaEvent_t init_done = nullptr, copied[2] = {}, consumed[2] = {};
};
RingRuntime g_ring[kMaxDevices];
std::mutex g_ring_mu;

int ring_runtime(RingRuntime** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_ring_mu);
    RingRuntime& r = g_ring[dev];
    if (!r.ready) {
        e = cudaStreamCreateWithFlags(&r.copy, cudaStreamNonBlocking);
        cudaEvent_t* evs[5] = {&r.init_done, &r.copied[0], &r.copied[1], &r.consumed[0], &r.consumed[1]};
        for (int x = 0; x < 5 && e == cudaSuccess; ++x)
            e = cudaEventCreateWithFlags(evs[x], cudaEventDisableTiming);
        if (e != cudaSuccess) return fail_cuda(e, "ring runtime set-up");
        r.ready = true;
    }
    *out = &r;
    return RA_OK;
}

struct EmuLayout {
    size_t kv_buf;      // one K (or V) receive buffer set: P ranks x B*H heads x C rows x d
    size_t off_k[2], off_v[2], off_o, off_part, off_lse, total;
};

EmuLayout emu_layout(int B, int H, int S, int d)
{
    EmuLayout L;
    const size_t rows = (size_t)B * H * S;
    L.kv_buf = ra::bwd::align256(rows * d * 2);
    size_t off = 0;
    for (int b = 0; b < 2; ++b) {
        L.off_k[b] = off; off += L.kv_buf;
        L.off_v[b] = off; off += L.kv_buf;
    }
    L.off_o = off; off += ra::bwd::align256(rows * d * 4);
    L.off_part = off; off += ra::bwd::align256(rows * d * 4);
    L.off_lse = off; off += ra::bwd::align256(rows * 4);
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

int ring_attn_fwd(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, ra_bf16* o, float* lse,
                  int B, int H, int S, int d, int P, int causal, float scale, void* stream)
{
    return fwd_impl(q, k, v, o, lse, B, H, H, S, d, P, causal, scale, stream);
}

int ring_attn_fwd_gqa(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, ra_bf16* o, float* lse,
                      int B, int H, int H_kv, int S, int d, int P, int causal, float scale,
                      void* stream)
{
    return fwd_impl(q, k, v, o, lse, B, H, H_kv, S, d, P, causal, scale, stream);
}

size_t ring_attn_fwd_f32_workspace_size(int B, int H, int H_kv, int S, int d)
{
    if (B <= 0 || H <= 0 || H_kv <= 0 || S <= 0 || d <= 0) return 0;
    const size_t q_elems = (size_t)B * H * S * d, kv_elems = (size_t)B * H_kv * S * d;
    return ra::bwd::align256(q_elems * 2) + 2 * ra::bwd::align256(kv_elems * 2);
}

int ring_attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                      int H, int H_kv, int S, int d, int P, int causal, float scale, void* workspace,
                      size_t workspace_bytes, void* stream)
{
    int rc = check_shape(B, H, S, d, P, causal, scale);
    if (rc != RA_OK) return rc;
    if (H_kv < 1 ? H != 0 : (H % H_kv) != 0) return RA_ERR_INVALID_ARG;
    if ((long long)B * H * S == 0) return RA_OK;
    if (!q || !k || !v || !o || !lse || !workspace) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RA_ERR_INVALID_ARG;
    if ((const void*)o == (const void*)k || (const void*)o == (const void*)v) return RA_ERR_INVALID_ARG;
    if (workspace_bytes < ring_attn_fwd_f32_workspace_size(B, H, H_kv, S, d)) return RA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st)) != RA_OK) return rc;
    const size_t q_elems = (size_t)B * H * S * d, kv_elems = (size_t)B * H_kv * S * d;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __nv_bfloat16* qb = reinterpret_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* kb = reinterpret_cast<__nv_bfloat16*>(ws + ra::bwd::align256(q_elems * 2));
    __nv_bfloat16* vb = reinterpret_cast<__nv_bfloat16*>(ws + ra::bwd::align256(q_elems * 2) +
                                                         ra::bwd::align256(kv_elems * 2));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long cap = (long long)st->num_sms * 16;
    const float* src[3] = {q, k, v};
    __nv_bfloat16* dst[3] = {qb, kb, vb};
    const size_t elems[3] = {q_elems, kv_elems, kv_elems};
    for (int x = 0; x < 3; ++x) {
        const long long n8 = (long long)(elems[x] / 8);   // d is 64 or 128
        long long blocks = (n8 + 255) / 256;
        if (blocks > cap) blocks = cap;
        ra::prof::Scope ps(ra::prof::kInConvert, s);
        ra::f32_to_bf16_kernel<<<(unsigned)blocks, 256, 0, s>>>(src[x], dst[x], n8);
        ps.done();
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda(e, "f32_to_bf16_kernel launch");
    }
    return fwd_impl(reinterpret_cast<const ra_bf16*>(qb), reinterpret_cast<const ra_bf16*>(kb),
                    reinterpret_cast<const ra_bf16*>(vb), nullptr, lse, B, H, H_kv, S, d, P, causal,
                    scale, stream, nullptr, nullptr, nullptr, nullptr, o);
}

int ring_attn_fwd_strided(const ra_bf16* q, const long long* q_strides, const ra_bf16* k,
                          const long long* k_strides, const ra_bf16* v, const long long* v_strides,
                          ra_bf16* o, const long long* o_strides, float* lse, int B, int H, int H_kv,
                          int S, int d, int P, int causal, float scale, void* stream)
{
    return fwd_impl(q, k, v, o, lse, B, H, H_kv, S, d, P, causal, scale, stream, q_strides, k_strides,
                    v_strides, o_strides);
}

size_t ring_attn_fwd_emulated_workspace_size(int B, int H, int S, int d)
{
    if (B <= 0 || H <= 0 || S <= 0 || d <= 0) return 0;
    return emu_layout(B, H, S, d).total;
}

int ring_attn_fwd_emulated(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, ra_bf16* o,
                           float* lse, int B, int H, int S, int d, int P, int causal, float scale,
                           void* workspace, size_t workspace_bytes, int overlap, void* stream)
{
    int rc = check_shape(B, H, S, d, P, causal, scale);
    if (rc != RA_OK) return rc;
    if (overlap != 0 && overlap != 1) return RA_ERR_INVALID_ARG;
    if ((long long)B * H * S == 0) return RA_OK;
    if (!q || !k || !v || !o || !lse || !workspace) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RA_ERR_INVALID_ARG;
    const EmuLayout lay = emu_layout(B, H, S, d);
    if (workspace_bytes < lay.total) return RA_ERR_INVALID_ARG;
    const int C = S / P;
    const long long pairs = (C + ra::fwd::kRowsPerCta - 1) / ra::fwd::kRowsPerCta;
    const long long grid = (long long)B * H * P * pairs;
    if (grid > 0x7fffffffll) return RA_ERR_UNSUPPORTED;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st)) != RA_OK) return rc;
    RingRuntime* rr = nullptr;
    if ((rc = ring_runtime(&rr)) != RA_OK) return rc;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ra_bf16* kbuf[2] = {reinterpret_cast<ra_bf16*>(ws + lay.off_k[0]), reinterpret_cast<ra_bf16*>(ws + lay.off_k[1])};
    ra_bf16* vbuf[2] = {reinterpret_cast<ra_bf16*>(ws + lay.off_v[0]), reinterpret_cast<ra_bf16*>(ws + lay.off_v[1])};
    float* o_run = reinterpret_cast<float*>(ws + lay.off_o);
    float* o_part = reinterpret_cast<float*>(ws + lay.off_part);
    float* lse_part = reinterpret_cast<float*>(ws + lay.off_lse);
    const int BH = B * H;
    const size_t chunk_bytes = (size_t)C * d * 2;          // one head's chunk
    const size_t rank_bytes = (size_t)BH * chunk_bytes;    // one rank's K (or V)
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t xs = overlap ? rr->copy : cs;             // the interconnect
    cudaError_t e = cudaSuccess;

    // Step 0 set-up: every rank holds its own chunk (K_i, V_i) in buffer 0.
    for (int i = 0; i < P && e == cudaSuccess; ++i) {
        e = cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(kbuf[0]) + (size_t)i * rank_bytes, chunk_bytes,
                              reinterpret_cast<const uint8_t*>(k) + (size_t)i * chunk_bytes,
                              (size_t)S * d * 2, chunk_bytes, BH, cudaMemcpyDeviceToDevice, cs);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(vbuf[0]) + (size_t)i * rank_bytes, chunk_bytes,
                                  reinterpret_cast<const uint8_t*>(v) + (size_t)i * chunk_bytes,
                                  (size_t)S * d * 2, chunk_bytes, BH, cudaMemcpyDeviceToDevice, cs);
    }
    if (e == cudaSuccess) e = cudaEventRecord(rr->init_done, cs);
    if (e != cudaSuccess) return fail_cuda(e, "ring set-up copies");

    CUtensorMap mq;
    bool r4q = false, r4kv = false;
    if ((rc = make_map(&mq, q, B, H, S, d, ra::contiguous_layout(H, S, d), ra::fwd::kBM, &r4q)) != RA_OK)
        return rc;
    for (int t = 0; t < P; ++t) {
        const int cur = t & 1, nxt = cur ^ 1;
        // Rotation for step t + 1 on the interconnect: rank i sends the
        // chunk it holds to rank (i + 1) % P, into the other buffer -- once
        // step t - 1 has finished reading that buffer.
        if (t + 1 < P) {
            if (t == 0) e = cudaStreamWaitEvent(xs, rr->init_done, 0);
            else e = cudaStreamWaitEvent(xs, rr->consumed[nxt], 0);
            for (int i = 0; i < P && e == cudaSuccess; ++i) {
                const size_t src = (size_t)i * rank_bytes, dst = (size_t)((i + 1) % P) * rank_bytes;
                e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(kbuf[nxt]) + dst,
                                    reinterpret_cast<uint8_t*>(kbuf[cur]) + src, rank_bytes,
                                    cudaMemcpyDeviceToDevice, xs);
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(vbuf[nxt]) + dst,
                                        reinterpret_cast<uint8_t*>(vbuf[cur]) + src, rank_bytes,
                                        cudaMemcpyDeviceToDevice, xs);
            }
            if (e == cudaSuccess) e = cudaEventRecord(rr->copied[nxt], xs);
            if (e != cudaSuccess) return fail_cuda(e, "ring rotation copies");
        }
        // Compute step t on the chunks each rank holds now.
        if (t > 0 && (e = cudaStreamWaitEvent(cs, rr->copied[cur], 0)) != cudaSuccess)
            return fail_cuda(e, "ring wait");
        CUtensorMap mk, mv;
        // receive buffers: [P * B, H, C, d], contiguous
        const ra::RowLayout lbuf = ra::contiguous_layout(H, C, d);
        if ((rc = make_map(&mk, kbuf[cur], P * B, H, C, d, lbuf, ra::fwd::kBN, &r4kv)) != RA_OK) return rc;
        if ((rc = make_map(&mv, vbuf[cur], P * B, H, C, d, lbuf, ra::fwd::kBN, &r4kv)) != RA_OK) return rc;
        ra::fwd::FwdParams prm;
        prm.rank4 = (r4q ? 1 : 0) | (r4kv ? 6 : 0);
        prm.o = nullptr;
        prm.lo = ra::contiguous_layout(H, S, d);
        prm.o32 = t == 0 ? o_run : o_part;          // step 0 starts the running result
        prm.lse = t == 0 ? lse : lse_part;
        prm.S = S;
        prm.P = P;
        prm.C = C;
        prm.causal = causal;
        prm.pairs_per_chunk = (int)pairs;
        prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
        prm.status = st->status;
        prm.wait_limit_ns = g_wait_limit_ns.load();
        prm.H = H;
        prm.group = 1;
        prm.step = t;
        prm.BH = BH;
        {
            ra::prof::Scope ps(ra::prof::kFwd, cs);
            if (d == 128)
                ra::fwd::ring_fwd_kernel<128><<<(unsigned)grid, ra::fwd::kThreads,
                                                ra::fwd::Cfg<128>::kSmemBytes, cs>>>(mq, mk, mv, prm);
            else
                ra::fwd::ring_fwd_kernel<64><<<(unsigned)grid, ra::fwd::kThreads,
                                               ra::fwd::Cfg<64>::kSmemBytes, cs>>>(mq, mk, mv, prm);
            ps.done();
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return fail_cuda(e, "ring step launch");
        if ((e = cudaEventRecord(rr->consumed[cur], cs)) != cudaSuccess) return fail_cuda(e, "ring event");
        if (t > 0) {
            // fold the step's partial into the running result (in place)
            rc = attn_merge_partials(o_run, lse, o_part, lse_part, o_run, lse, B, H, S, d, stream);
            if (rc != RA_OK) return rc;
        }
    }
    // O (fp32, normalized) -> bf16
    const long long n8 = (long long)((size_t)BH * S * d / 8);
    long long cb = (n8 + 255) / 256;
    const long long cap = (long long)st->num_sms * 16;
    if (cb > cap) cb = cap;
    if (d == 128)
        ra::dq_convert_kernel<128, false><<<(unsigned)cb, 256, 0, cs>>>(o_run, reinterpret_cast<__nv_bfloat16*>(o),
                                                                ra::contiguous_layout(H, S, d), n8, H, S);
    else
        ra::dq_convert_kernel<64, false><<<(unsigned)cb, 256, 0, cs>>>(o_run, reinterpret_cast<__nv_bfloat16*>(o),
                                                               ra::contiguous_layout(H, S, d), n8, H, S);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail_cuda(e, "ring output convert");
    return RA_OK;
}

}  // extern "C"

namespace {

// ---------------------------------------------------------------------------
// Ulysses layout on one GPU: P logical ranks, two all-to-alls
// ---------------------------------------------------------------------------
// ("Context Parallelism" guide, section 3 "Ulysses (DeepSpeed)", steps 1-4;
// "Training Long-Context Models Without OOM: Ring Attention", section "Ring
// Attention vs. DeepSpeed Ulysses (All-to-All)".)  Rank i starts with tokens
// [iC, (i+1)C) of every head.  An all-to-all redistributes by head: rank r
// receives, from every rank i, the tokens of chunk i for its heads
// [r H/P, (r+1) H/P) (and key/value heads [r H_kv/P, (r+1) H_kv/P)), so it
// holds full sequences of H/P heads.  Each rank then computes full-sequence
// attention for its heads, and a second all-to-all sends each rank's O and
// LSE rows of chunk i back to rank i.
//
// Workspace: the ranks' receive buffers, [P, B, H/P, S, d] for q and O,
// [P, B, H_kv/P, S, d] for k and v (bf16), and [P, B, H/P, S] fp32 for LSE.
struct UlyssesLayout {
    size_t off_q, off_k, off_v, off_o, off_lse, total;
};

UlyssesLayout ulysses_layout(int B, int H, int H_kv, int S, int d)
{
    UlyssesLayout L;
    const size_t q_elems = (size_t)B * H * S * d, kv_elems = (size_t)B * H_kv * S * d;
    size_t off = 0;
    L.off_q = off; off += ra::bwd::align256(q_elems * 2);
    L.off_k = off; off += ra::bwd::align256(kv_elems * 2);
    L.off_v = off; off += ra::bwd::align256(kv_elems * 2);
    L.off_o = off; off += ra::bwd::align256(q_elems * 2);
    L.off_lse = off; off += ra::bwd::align256((size_t)B * H * S * 4);
    L.total = off;
    return L;
}

// One all-to-all over a [B, heads, S, w]-element tensor held as P sequence
// shards: block (rank i -> rank r) is chunk i of heads [r hp, (r+1) hp) of
// every batch.  to_heads: sequence shards (the caller's tensor) -> head
// shards ([P, B, hp, S, w] buffer); otherwise the way back.  One 2-D copy
// per (batch, source rank, destination rank): P^2 B messages.
cudaError_t all_to_all(void* seq, void* heads_buf, int B, int heads, int S, int w, size_t elem, int P,
                       bool to_heads, cudaStream_t s)
{
    const int hp = heads / P, C = S / P;
    const size_t pitch = (size_t)S * w * elem, width = (size_t)C * w * elem;
    cudaError_t e = cudaSuccess;
    for (int r = 0; r < P && e == cudaSuccess; ++r)
        for (int b = 0; b < B && e == cudaSuccess; ++b)
            for (int i = 0; i < P && e == cudaSuccess; ++i) {
                uint8_t* sp = static_cast<uint8_t*>(seq) +
                              (((size_t)b * heads + (size_t)r * hp) * S + (size_t)i * C) * w * elem;
                uint8_t* hb = static_cast<uint8_t*>(heads_buf) +
                              ((((size_t)r * B + b) * hp) * S + (size_t)i * C) * w * elem;
                e = to_heads ? cudaMemcpy2DAsync(hb, pitch, sp, pitch, width, hp, cudaMemcpyDeviceToDevice, s)
                             : cudaMemcpy2DAsync(sp, pitch, hb, pitch, width, hp, cudaMemcpyDeviceToDevice, s);
            }
    return e;
}

}  // namespace

extern "C" {

size_t ring_attn_fwd_ulysses_workspace_size(int B, int H, int H_kv, int S, int d)
{
    if (B <= 0 || H <= 0 || H_kv <= 0 || S <= 0 || d <= 0) return 0;
    return ulysses_layout(B, H, H_kv, S, d).total;
}

int ring_attn_fwd_ulysses_emulated(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, ra_bf16* o,
                                   float* lse, int B, int H, int H_kv, int S, int d, int P, int causal,
                                   float scale, void* workspace, size_t workspace_bytes, void* stream)
{
    int rc = check_shape(B, H, S, d, P, causal, scale);
    if (rc != RA_OK) return rc;
    if (H_kv < 1 ? H != 0 : (H % H_kv) != 0) return RA_ERR_INVALID_ARG;
    if ((long long)B * H * S == 0) return RA_OK;
    // every rank needs whole heads: P must divide the query and key/value head counts
    if (H % P != 0 || H_kv % P != 0) return RA_ERR_UNSUPPORTED;
    if (!q || !k || !v || !o || !lse || !workspace) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RA_ERR_INVALID_ARG;
    const UlyssesLayout lay = ulysses_layout(B, H, H_kv, S, d);
    if (workspace_bytes < lay.total) return RA_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // step 2: all-to-all on Q, K and V (sequence shards -> head shards)
    cudaError_t e = all_to_all(const_cast<ra_bf16*>(q), ws + lay.off_q, B, H, S, d, 2, P, true, cs);
    if (e == cudaSuccess) e = all_to_all(const_cast<ra_bf16*>(k), ws + lay.off_k, B, H_kv, S, d, 2, P, true, cs);
    if (e == cudaSuccess) e = all_to_all(const_cast<ra_bf16*>(v), ws + lay.off_v, B, H_kv, S, d, 2, P, true, cs);
    if (e != cudaSuccess) return fail_cuda(e, "Ulysses all-to-all (q, k, v)");
    // step 3: every rank's full-sequence attention for its heads; the ranks'
    // buffers together are P * B batches of H / P heads, one launch
    rc = fwd_impl(reinterpret_cast<const ra_bf16*>(ws + lay.off_q), reinterpret_cast<const ra_bf16*>(ws + lay.off_k),
                  reinterpret_cast<const ra_bf16*>(ws + lay.off_v), reinterpret_cast<ra_bf16*>(ws + lay.off_o),
                  reinterpret_cast<float*>(ws + lay.off_lse), P * B, H / P, H_kv / P, S, d, 1, causal, scale,
                  stream);
    if (rc != RA_OK) return rc;
    // step 4: all-to-all on the output (head shards -> sequence shards)
    e = all_to_all(o, ws + lay.off_o, B, H, S, d, 2, P, false, cs);
    if (e == cudaSuccess) e = all_to_all(lse, ws + lay.off_lse, B, H, S, 1, 4, P, false, cs);
    if (e != cudaSuccess) return fail_cuda(e, "Ulysses all-to-all (O, LSE)");
    return RA_OK;
}

size_t ring_attn_bwd_workspace_size(int B, int H, int S, int d)
{
    if (B <= 0 || H <= 0 || S <= 0 || d <= 0) return 0;
    return ra::bwd::workspace_bytes(B, H, S, d);
}

int ring_attn_bwd(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, const ra_bf16* o,
                  const float* lse, const ra_bf16* dO, ra_bf16* dq, ra_bf16* dk, ra_bf16* dv,
                  int B, int H, int S, int d, int P, int causal, float scale, void* workspace,
                  size_t workspace_bytes, void* stream)
{
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, H, S, d, P, causal, scale, workspace,
                    workspace_bytes, stream);
}

int ring_attn_bwd_gqa(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, const ra_bf16* o,
                      const float* lse, const ra_bf16* dO, ra_bf16* dq, ra_bf16* dk, ra_bf16* dv,
                      int B, int H, int H_kv, int S, int d, int P, int causal, float scale,
                      void* workspace, size_t workspace_bytes, void* stream)
{
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, S, d, P, causal, scale, workspace,
                    workspace_bytes, stream);
}

int ring_attn_bwd_strided(const ra_bf16* q, const long long* q_strides, const ra_bf16* k,
                          const long long* k_strides, const ra_bf16* v, const long long* v_strides,
                          const ra_bf16* o, const long long* o_strides, const float* lse,
                          const ra_bf16* dO, const long long* do_strides, ra_bf16* dq,
                          const long long* dq_strides, ra_bf16* dk, const long long* dk_strides,
                          ra_bf16* dv, const long long* dv_strides, int B, int H, int H_kv, int S,
                          int d, int P, int causal, float scale, void* workspace,
                          size_t workspace_bytes, void* stream)
{
    const long long* const strides[8] = {q_strides, k_strides, v_strides, o_strides,
                                         do_strides, dq_strides, dk_strides, dv_strides};
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, S, d, P, causal, scale, workspace,
                    workspace_bytes, stream, strides);
}

}  // extern "C"

namespace {

// strides: NULL, or 8 stride triples (or NULLs) for q, k, v, o, dO, dq, dk, dv.
int bwd_impl(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, const ra_bf16* o,
             const float* lse, const ra_bf16* dO, ra_bf16* dq, ra_bf16* dk, ra_bf16* dv, int B,
             int H, int H_kv, int S, int d, int P, int causal, float scale, void* workspace,
             size_t workspace_bytes, void* stream, const long long* const* strides)
{
    int rc = check_shape(B, H, S, d, P, causal, scale);
    if (rc != RA_OK) return rc;
    if (H_kv < 1 ? H != 0 : (H % H_kv) != 0) return RA_ERR_INVALID_ARG;
    if ((long long)B * H * S == 0) return RA_OK;   // empty: nothing to launch or read
    auto st_of = [&](int x) { return strides ? strides[x] : nullptr; };
    ra::RowLayout lq = layout_from(st_of(0), H, S, d), lk = layout_from(st_of(1), H_kv, S, d),
                  lv = layout_from(st_of(2), H_kv, S, d), lo = layout_from(st_of(3), H, S, d),
                  ldo = layout_from(st_of(4), H, S, d), ldq = layout_from(st_of(5), H, S, d),
                  ldk = layout_from(st_of(6), H_kv, S, d), ldv = layout_from(st_of(7), H_kv, S, d);
    if (!layout_ok(lq, B, H, S) || !layout_ok(lk, B, H_kv, S) || !layout_ok(lv, B, H_kv, S) ||
        !layout_ok(lo, B, H, S) || !layout_ok(ldo, B, H, S) || !layout_ok(ldq, B, H, S) ||
        !layout_ok(ldk, B, H_kv, S) || !layout_ok(ldv, B, H_kv, S))
        return RA_ERR_INVALID_ARG;
    if ((long long)B * H * S == 0) return RA_OK;
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace)
        return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RA_ERR_INVALID_ARG;
    if (workspace_bytes < ra::bwd::workspace_bytes(B, H, S, d)) return RA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    rc = device_state(&st);
    if (rc != RA_OK) return rc;
    ra::bwd::Launch L;
    L.q = q; L.k = k; L.v = v; L.o = o; L.lse = lse; L.dO = dO;
    L.dq = dq; L.dk = dk; L.dv = dv;
    L.lq = lq; L.lk = lk; L.lv = lv; L.lo = lo; L.ldo = ldo; L.ldq = ldq; L.ldk = ldk; L.ldv = ldv;
    L.B = B; L.H = H; L.H_kv = H_kv; L.S = S; L.d = d; L.P = P; L.causal = causal; L.scale = scale;
    L.workspace = workspace;
    L.status = st->status;
    L.num_sms = st->num_sms;
    L.wait_limit_ns = g_wait_limit_ns.load();
    L.stream = static_cast<cudaStream_t>(stream);
    L.encode = [](CUtensorMap* m, const void* p, int B_, int heads, int S_, int d_, ra::RowLayout lay,
                  int rows, bool* rank4) { return make_map(m, p, B_, heads, S_, d_, lay, rows, rank4); };
    L.encode_rows = [](CUtensorMap* m, const float* p, int BH, int S_) {
        return make_row_map(m, p, BH, S_);
    };
    L.encode_acc = [](CUtensorMap* m, float* p, int BH, int S_, int d_) {
        return make_acc_map(m, p, BH, S_, d_);
    };
    cudaError_t e = cudaSuccess;
    rc = ra::bwd::launch(L, &e);
    if (rc == RA_ERR_CUDA) return fail_cuda(e, "ring_bwd launch");
    return rc;
}

}  // namespace

extern "C" {

int ring_attn_bwd_noalloc(const ra_bf16* q, const ra_bf16* k, const ra_bf16* v, const ra_bf16* o,
                          const float* lse, const ra_bf16* dO, ra_bf16* dq, ra_bf16* dk, ra_bf16* dv,
                          int B, int H, int S, int d, int P, int causal, float scale, void* stream)
{
    int rc = check_shape(B, H, S, d, P, causal, scale);
    if (rc != RA_OK) return rc;
    if ((long long)B * H * S == 0) return RA_OK;
    if (ra::bwd::workspace_bytes(B, H, S, d) > RING_ATTN_NOALLOC_SCRATCH_BYTES) return RA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != RA_OK) return rc;
    return ring_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, S, d, P, causal, scale, scratch,
                         RING_ATTN_NOALLOC_SCRATCH_BYTES, stream);
}

int attn_merge_partials(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                        float* o_out, float* lse_out, int B, int H, int S, int d, void* stream)
{
    if (B < 0 || H < 0 || S < 0 || d < 1) return RA_ERR_INVALID_ARG;
    const long long rows = (long long)B * H * S;
    if (rows == 0) return RA_OK;
    if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out) return RA_ERR_INVALID_ARG;
    if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(o_out) ||
        (reinterpret_cast<uintptr_t>(lse_a) & 3u) || (reinterpret_cast<uintptr_t>(lse_b) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse_out) & 3u))
        return RA_ERR_INVALID_ARG;
    // Only the documented in-place form may alias.
    if (o_out == o_b || lse_out == lse_b || (const void*)o_out == (const void*)lse_a)
        return RA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != RA_OK) return rc;
    const long long warps_needed = rows;
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = (long long)st->num_sms * 16;
    if (blocks > cap) blocks = cap;
    ra::prof::Scope ps(ra::prof::kMerge, static_cast<cudaStream_t>(stream));
    ra::merge_partials_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        o_a, lse_a, o_b, lse_b, o_out, lse_out, rows, d);
    ps.done();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "merge_partials_kernel launch");
    return RA_OK;
}

int ring_attn_trace_visits(int* buf, long long capacity)
{
    if (capacity < 0 || (buf == nullptr) != (capacity == 0)) return RA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(buf) & 15u) return RA_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != RA_OK) return rc;
    const ra::VisitTrace t{buf, capacity};
    const cudaError_t e = cudaMemcpyToSymbol(ra::g_visit_trace, &t, sizeof(t));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyToSymbol(visit trace)");
    return RA_OK;
}

int ring_attn_profile_enable(int on)
{
    ra::prof::g_on.store(on ? 1 : 0);
    return RA_OK;
}

int ring_attn_profile_reset(void)
{
    ra::prof::reset();
    return RA_OK;
}

int ring_attn_profile_read(const char* kernel, double* total_ms, long long* launches)
{
    if (!kernel || !total_ms || !launches) return RA_ERR_INVALID_ARG;
    ra::prof::collect();
    for (int k = 0; k < ra::prof::kKinds; ++k) {
        if (std::strcmp(kernel, ra::prof::kind_name(k)) == 0) {
            std::lock_guard<std::mutex> lock(ra::prof::g_mu);
            *total_ms = ra::prof::g_ms[k];
            *launches = ra::prof::g_count[k];
            return RA_OK;
        }
    }
    return RA_ERR_INVALID_ARG;
}

int ring_attn_check_status(void* stream)
{
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != RA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    uint32_t word = 0;
    e = cudaMemcpyAsync(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(st->status, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "status read");
    return word ? RA_ERR_DEVICE_TIMEOUT : RA_OK;
}

}  // extern "C"
