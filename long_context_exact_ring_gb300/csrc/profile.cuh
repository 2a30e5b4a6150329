// profile.cuh -- optional per-kernel timing of the library's own launches.
//
// When enabled, every kernel launch is bracketed by a pair of CUDA events
// recorded on the launch stream; ring_attn_profile_read() synchronizes on
// them and returns, per kernel, the number of launches and the summed
// device time since the last reset.  Disabled (the default) it costs one
// relaxed atomic load per launch.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

namespace ra {
namespace prof {

enum Kind : int { kFwd = 0, kBwdMain, kBwdPrep, kDqConvert, kMerge, kInConvert, kKinds };

inline const char* kind_name(int k)
{
    static const char* names[kKinds] = {"ring_fwd_kernel", "ring_bwd_kernel", "bwd_prep_kernel",
                                        "dq_convert_kernel", "merge_partials_kernel",
                                        "f32_to_bf16_kernel"};
    return (k >= 0 && k < kKinds) ? names[k] : "";
}

struct Rec {
    int kind;
    cudaEvent_t a, b;
};

inline std::atomic<int> g_on{0};
inline std::mutex g_mu;
inline std::vector<Rec> g_pending;
inline std::vector<cudaEvent_t> g_pool;
inline double g_ms[kKinds] = {};
inline long long g_count[kKinds] = {};

inline cudaEvent_t take_event()
{
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Brackets one launch: construct before the launch, call done() after it.
struct Scope {
    int kind = -1;
    cudaEvent_t a = nullptr, b = nullptr;
    cudaStream_t s = nullptr;
    Scope(int k, cudaStream_t stream)
    {
        if (!g_on.load(std::memory_order_relaxed)) return;
        std::lock_guard<std::mutex> lock(g_mu);
        a = take_event();
        b = take_event();
        if (!a || !b) return;
        kind = k;
        s = stream;
        cudaEventRecord(a, s);
    }
    void done()
    {
        if (kind < 0) return;
        cudaEventRecord(b, s);
        std::lock_guard<std::mutex> lock(g_mu);
        g_pending.push_back({kind, a, b});
        kind = -1;
    }
};

// Fold finished records into the totals (synchronizes on their events).
inline void collect()
{
    std::lock_guard<std::mutex> lock(g_mu);
    for (const Rec& r : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
            g_ms[r.kind] += ms;
            g_count[r.kind] += 1;
        }
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_pending.clear();
}

inline void reset()
{
    collect();
    std::lock_guard<std::mutex> lock(g_mu);
    for (int k = 0; k < kKinds; ++k) {
        g_ms[k] = 0.0;
        g_count[k] = 0;
    }
}

}  // namespace prof
}  // namespace ra
