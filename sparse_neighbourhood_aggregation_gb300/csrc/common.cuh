// Internal helpers shared by the libgnn translation units (never by the
// CPU oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gnn.h"

namespace gnn {

// ---------------------------------------------------------------- host side

// Count every kernel launch of the library (gnn_launch_count).
void note_launch(int n = 1);

// Record the first error of a CUDA call; returns GNN_ERR_CUDA on failure.
gnn_status cuda_status(cudaError_t e);

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Edges per run of the degree-aware edge-run schedule (aggregation and
// attention kernels); the prepared graph stores each run's first row.
#ifndef GNN_RUN_EDGES
#define GNN_RUN_EDGES 64
#endif
constexpr int32_t kRunEdges = GNN_RUN_EDGES;
// Edges per span of the edge-span aggregation kernel: a power of two >= 64
// chosen from the graph's size, so that a graph has at least ~16 resident
// waves of spans (longer spans amortise each warp's start-up and cut fewer
// rows; shorter ones keep small graphs busy).  The prepared graph stores each
// span's first edge.
#ifndef GNN_SPAN_EDGES
#define GNN_SPAN_EDGES 0   // 0: by graph size; otherwise fixed
#endif
inline int32_t span_shift(int64_t nnz) {
    if (GNN_SPAN_EDGES > 0) {
        int32_t k = 5;
        while ((1 << k) < GNN_SPAN_EDGES) ++k;
        return k;
    }
    return nnz >= ((int64_t)1 << 24) ? 8 : nnz >= ((int64_t)1 << 23) ? 7 : 6;
}
inline int32_t span_edges(int64_t nnz) { return 1 << span_shift(nnz); }
inline int64_t n_spans_of(int64_t nnz) { return (nnz + span_edges(nnz) - 1) / span_edges(nnz); }
// A row of degree > span_edges is cut into one piece per span it touches;
// its pieces are summed in chunks of kFixChunk, one work item per chunk.
constexpr int32_t kFixChunk = 16;
inline int64_t span_item_cap(int64_t nnz) {
    return nnz / (span_edges(nnz) + 1) + 2 * n_spans_of(nnz) / kFixChunk + 1;
}

inline int64_t n_runs(int64_t nnz, int32_t E) {
    int64_t n = (nnz + E - 1) / E;
    return n > 0 ? n : 1;
}

// Device error word (one per device, library static).  Kernels set it with
// atomicCAS from 0 so the first failure is kept.
int32_t *device_error_word();

// Number of SMs of the current device (cached).
int sm_count();

// cudaFuncSetAttribute(fn, attr, value) once per (kernel, current device,
// attribute, value): a kernel attribute belongs to a device's context, so a
// process that drives several GPUs sets it on each before launching there.
cudaError_t func_attr(const void *fn, cudaFuncAttribute attr, int value);

#define GNN_LAUNCH_CHECK()                                        \
    do {                                                          \
        cudaError_t e__ = cudaGetLastError();                     \
        if (e__ != cudaSuccess) return ::gnn::cuda_status(e__);   \
    } while (0)

// Carve sub-buffers out of a caller-provided byte buffer (256-byte aligned).
struct Carver {
    char *base;
    size_t used = 0;
    explicit Carver(void *b) : base(static_cast<char *>(b)) {}
    template <class T>
    T *take(size_t count) {
        T *p = reinterpret_cast<T *>(base ? base + used : nullptr);
        used = round_up(used + count * sizeof(T), 256);
        return p;
    }
};

// ---------------------------------------------------------------- device side

__device__ __forceinline__ void set_device_error(int32_t *word, int32_t code) {
    atomicCAS(word, 0, code);
}

// 16-byte read-only load through the non-coherent path.
__device__ __forceinline__ uint4 ldg16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// 16-byte load that bypasses L1 (data written by other CTAs of this launch).
__device__ __forceinline__ uint4 ldcg16(const void *p) {
    return __ldcg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Unpack a 16-byte chunk to fp32: 4 floats (fp32) or 8 floats (bf16).
template <class T>
struct Chunk;

template <>
struct Chunk<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *o) {
        o[0] = __uint_as_float(v.x);
        o[1] = __uint_as_float(v.y);
        o[2] = __uint_as_float(v.z);
        o[3] = __uint_as_float(v.w);
    }
};

template <>
struct Chunk<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *o) {
        o[0] = bf16lo(v.x); o[1] = bf16hi(v.x);
        o[2] = bf16lo(v.y); o[3] = bf16hi(v.y);
        o[4] = bf16lo(v.z); o[5] = bf16hi(v.z);
        o[6] = bf16lo(v.w); o[7] = bf16hi(v.w);
    }
};

// Order-preserving key of an fp32 value (IO-aware GNN layers, Appendix D.1):
// negative values have every bit inverted, non-negative values get the sign
// bit set; unsigned comparison of keys then orders the floats (-0 < +0).
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Inverse of order_key.
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// 2^x by the hardware approximation (ex2.approx.ftz; 2^-inf = +0)
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (Blackwell f32x2 instructions): d += a * b and a + b on
// two lanes of a 64-bit register pair.
__device__ __forceinline__ uint64_t pk2(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &x, float &y) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}


}  // namespace gnn
