// trace.cuh -- optional record of the ring order the kernels walk.
//
// Off by default: the descriptor below is {NULL, 0} until
// ring_attn_trace_visits() sets it, and every kernel reads it once per CTA.
// When it is set, the TMA producer thread of each CTA of ring_fwd_kernel and
// ring_bwd_kernel writes, into the CTA's own slot of the buffer, one entry
// per ring visit -- each time its stream of tiles enters a new chunk -- so
// that a test can compare the order the kernels really follow with the ring
// schedule ("Context Parallelism" guide, section 2, "How It Works": at step
// t query chunk i meets KV chunk (i - t) mod P; causal attention skips
// chunks above the diagonal).
//
// Slot of CTA x: (P + 1) entries of kTraceInts ints at buf + x (P + 1) kTraceInts.
//   entry 0 (header)
//     forward : {b H + h, query chunk i, first query row, visits, ring step
//                of a one-step launch or -1, tiles in total, 0, 0}
//     backward: {b H_kv + kv head, key chunk j, key tile, visits, tiles in
//                total, query heads per key/value head, 0, 0}
//   entries 1 .. visits, in the order visited
//     forward : {step t, key chunk j, kind, tiles, first key, last tile's
//                first key, 0, 0}
//     backward: {query chunk i, step t = (i - j) mod P, kind, tiles, first
//                query, last tile's first query, 0, 0}
//   kind: 0 when the chunk is the CTA's own (i == j), 1 otherwise.
// The backward records the query tiles of the first query head of a group;
// the other heads of the group repeat the same sequence.  A slot that does
// not fit the buffer's capacity is not written.
#pragma once

#include <stdint.h>

namespace ra {

struct VisitTrace {
    int* buf;
    long long cap;   // ints
};

__device__ VisitTrace g_visit_trace;

constexpr int kTraceInts = 8;

// This CTA's slot, or NULL when tracing is off or the slot does not fit.
__device__ __forceinline__ int* trace_slot(int P)
{
    const VisitTrace t = g_visit_trace;
    if (t.buf == nullptr) return nullptr;
    const long long per = (long long)(P + 1) * kTraceInts;
    if ((long long)(blockIdx.x + 1) * per > t.cap) return nullptr;
    return t.buf + (long long)blockIdx.x * per;
}

__device__ __forceinline__ void trace_put(int* e, int a, int b, int c, int d, int f, int g)
{
    e[0] = a; e[1] = b; e[2] = c; e[3] = d; e[4] = f; e[5] = g; e[6] = 0; e[7] = 0;
}

}  // namespace ra
