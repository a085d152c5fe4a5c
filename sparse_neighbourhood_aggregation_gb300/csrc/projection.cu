// Step a3: dense projection C = H W on the 5th-generation tensor cores.
//
// IO-aware GNN layers, Section 2.2 (i) and footnote 2: the node-wise linear
// map of a GNN layer is an ordinary dense GEMM (C = H W, H [n, F_in],
// W [F_in, F_out]); the GATv2 layer (Section 2.2 (iii)) projects with it
// before the fused edge pass.
//
// GB300 design (bf16 in, fp32 accumulation in TMEM, bf16 out).  The shapes
// of a GNN layer make this GEMM HBM-bound (F_in, F_out <= 256, n ~ 10^6):
// the whole of W stays in shared memory and each CTA streams 128-row tiles of
// H through it.  A persistent grid (one CTA per SM) runs three roles:
//   warp 0  TMA producer: 128 x 64 bf16 boxes of H (128-byte swizzle) into
//           a ring of shared-memory stages;
//   warp 1  MMA issuer: allocates TMEM, one elected thread issues
//           tcgen05.mma (M = 128, N = F_out, K = 16) into one of two TMEM
//           accumulators and commits each stage back to the producer;
//   warps 2-5 epilogue: tcgen05.ld of its 32-lane quarter of the
//           accumulator, fp32 -> bf16 (round to nearest even), stores; the
//           optional GATv2 per-node linear part sum_d coef_d C[i, hD + d]
//           is formed here from the rounded values, so C is not read again.
// The accumulators are double-buffered, so the epilogue of one tile
// overlaps the MMAs of the next.  W is transposed into the K-major swizzled
// operand layout once per CTA.  Every mbarrier wait is bounded: a wait that
// runs out sets the device error word (GNN_ERR_TIMEOUT), the CTA stops,
// waits (bounded) for its copies and MMAs in flight and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "async.cuh"
#include "common.cuh"
#include "tcgen05.cuh"

namespace gnn {

namespace {

constexpr int kBM = 128;                    // tile rows (MMA M)
constexpr int kBK = 64;                     // K per stage: 128 bytes of bf16
constexpr int kStageBytes = kBM * kBK * 2;  // 16 KB
constexpr int kMaxStages = 8;
constexpr int kThreads = 192;               // 6 warps

struct Bars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t bail;
};

// Wait for the phase of parity `parity` of barrier b; false if the CTA is
// bailing out or the wait ran out of time (then the CTA bails out).
__device__ __noinline__ bool mbar_wait(uint64_t *b, uint32_t parity, Bars *bars, int32_t *err) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_test(b, parity)) return true;
        if ((i & 255) == 255) {
            if (*reinterpret_cast<volatile int32_t *>(&bars->bail)) return false;
            const uint64_t t = globaltimer_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > kWaitLimitNs) {
                atomicExch(&bars->bail, 1);
                set_device_error(err, GNN_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
        : "memory");
}

struct ProjArgs {
    const __nv_bfloat16 *W;  // [Fi, Fo]
    __nv_bfloat16 *C;        // [n, Fo]
    const float *lin_coef;   // [Fo] or null: per-node linear parts
    float *lin_out;          // [n, lin_ld] (first `heads` columns written)
    int64_t ldc;             // C row stride (elements)
    int64_t lin_ld;          // lin_out row stride (floats)
    int64_t n;
    int32_t Fi, Fo;
    int32_t heads, D;
    int32_t stages;
    int32_t acc_cols;        // TMEM columns per accumulator (power of two >= Fo)
    int32_t *err;
};

__global__ void __launch_bounds__(kThreads, 1) k_proj_tc(const __grid_constant__ CUtensorMap tmH, ProjArgs p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned operand region: A ring, then W^T k-blocks
    unsigned char *base = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~(uintptr_t)1023);
    unsigned char *sA = base;
    unsigned char *sB = sA + (size_t)p.stages * kStageBytes;
    const int KB = p.Fi / kBK;
    Bars *bars = reinterpret_cast<Bars *>(sB + (size_t)KB * p.Fo * 128);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_tiles = (p.n + kBM - 1) / kBM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tfull[b], 1);
            mbar_init(&bars->tempty[b], 4 * 32);
        }
        mbar_init(&bars->drain, 1);
        bars->bail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(su32(&bars->tmem_base)), "r"(2 * p.acc_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // W^T into the K-major swizzled layout: k-block kb, row n, 16-byte chunk c
    // (k = 64 kb + 8 c .. +8) at sB + kb*Fo*128 + n*128 + ((c ^ (n & 7)) * 16).
    {
        const int nb8 = p.Fo / 8, kb8 = p.Fi / 8;
        for (int blk = threadIdx.x; blk < nb8 * kb8; blk += kThreads) {
            const int n0 = (blk % nb8) * 8, k0 = (blk / nb8) * 8;
            uint4 rows[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                rows[i] = __ldg(reinterpret_cast<const uint4 *>(p.W + (int64_t)(k0 + i) * p.Fo + n0));
            const uint16_t *rv = reinterpret_cast<const uint16_t *>(rows);
            const int kb = k0 / kBK, c = (k0 % kBK) / 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = (uint32_t)rv[(2 * q) * 8 + j] | ((uint32_t)rv[(2 * q + 1) * 8 + j] << 16);
                const int nn = n0 + j;
                *reinterpret_cast<uint4 *>(sB + (size_t)kb * p.Fo * 128 + (size_t)nn * 128 +
                                           (size_t)((c ^ (nn & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmH)) : "memory");
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&bars->empty[stage], phase ^ 1u, bars, p.err)) { ok = false; break; }
                    mbar_expect_tx(&bars->full[stage], kStageBytes);
                    tma_load_2d(sA + (size_t)stage * kStageBytes, &tmH, kb * kBK, (int32_t)(t * kBM),
                                &bars->full[stage]);
                    ++issued;
                    if (++stage == p.stages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // copies still in flight land before the CTA leaves: wait for
                // the last issue on every stage (bounded; no bail check)
                const int64_t k0 = issued > p.stages ? issued - p.stages : 0;
                for (int64_t k = k0; k < issued; ++k) {
                    const int s = (int)(k % p.stages);
                    const uint32_t ph = (uint32_t)((k / p.stages) & 1);
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_test(&bars->full[s], ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = bf16_idesc(kBM, p.Fo);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, bars, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * p.acc_cols);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&bars->full[stage], phase, bars, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = su32(sA + (size_t)stage * kStageBytes);
                    const uint32_t b0 = su32(sB + (size_t)kb * p.Fo * 128);
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks)
                        umma_bf16(d_tmem, sw128_desc(a0 + ks * 32), sw128_desc(b0 + ks * 32), idesc,
                                  (kb | ks) != 0 ? 1u : 0u);
                    umma_commit(&bars->empty[stage]);
                    if (++stage == p.stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&bars->tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // every MMA issued has completed before TMEM is released
            umma_commit(&bars->drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(&bars->drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row_in_tile = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            // the warp-wide tcgen05.ld below needs every lane on the same path
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->tfull[acc], acc_phase, bars, p.err));
            if (!ok) break;
            tc_fence_after();
            const int64_t row = t * kBM + row_in_tile;
            const bool in = row < p.n;
            float lin = 0.f;
            for (int c0 = 0; c0 < p.Fo; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.acc_cols + c0), v);
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const __nv_bfloat162 b2 =
                        __floats2bfloat162_rn(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
                    pk[k] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                if (in) {
                    // F_out may end half way through the 32-column chunk
                    uint4 *dst = reinterpret_cast<uint4 *>(p.C + row * p.ldc + c0);
                    const int nq = min(32, p.Fo - c0) / 8;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (k < nq) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
                if (p.lin_coef) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        lin = fmaf(__ldg(p.lin_coef + c0 + 2 * k), bf16lo(pk[k]), lin);
                        lin = fmaf(__ldg(p.lin_coef + c0 + 2 * k + 1), bf16hi(pk[k]), lin);
                    }
                    if (((c0 + 32) % p.D) == 0) {
                        if (in) p.lin_out[row * p.lin_ld + (c0 + 32) / p.D - 1] = lin;
                        lin = 0.f;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bars->tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * p.acc_cols));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

}  // namespace

// Shapes the tensor-core path covers.
bool projection_tc_supported(int64_t n, int32_t Fi, int32_t Fo) {
    return n > 0 && Fi >= kBK && Fi <= 256 && Fi % kBK == 0 && Fo >= 16 && Fo <= 256 && Fo % 16 == 0 &&
           n < ((int64_t)1 << 31);
}

// C = H W (bf16) on tcgen05, C rows ldc elements apart.  lin_coef (device
// [Fo], may be null): also write lin_out[i * lin_ld + h] =
// sum_{d < D} lin_coef[hD + d] C[i, hD + d] (C as rounded to bf16),
// D % 32 == 0.
gnn_status projection_tc_lin(const void *H, int64_t n, int32_t Fi, const void *W, int32_t Fo, void *C,
                             int64_t ldc, const float *lin_coef, int32_t heads, int32_t D, float *lin_out,
                             int64_t lin_ld, cudaStream_t s) {
    if (!projection_tc_supported(n, Fi, Fo)) return GNN_ERR_UNSUPPORTED;
    if (lin_coef && (D % 32 || heads * D != Fo || !lin_out)) return GNN_ERR_UNSUPPORTED;
    if (!aligned16(H) || !aligned16(W) || !aligned16(C) || ldc < Fo || ldc % 8) return GNN_ERR_UNSUPPORTED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return GNN_ERR_UNSUPPORTED;
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;

    CUtensorMap tm;
    cuuint64_t gdim[2] = {(cuuint64_t)Fi, (cuuint64_t)n};
    cuuint64_t gstride[1] = {(cuuint64_t)Fi * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(H), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return GNN_ERR_CUDA;

    ProjArgs p{};
    p.W = static_cast<const __nv_bfloat16 *>(W);
    p.C = static_cast<__nv_bfloat16 *>(C);
    p.lin_coef = lin_coef;
    p.lin_out = lin_out;
    p.ldc = ldc;
    p.lin_ld = lin_ld;
    p.n = n;
    p.Fi = Fi;
    p.Fo = Fo;
    p.heads = heads;
    p.D = D > 0 ? D : 32;
    p.err = err;
    int acc_cols = 32;
    while (acc_cols < Fo) acc_cols *= 2;
    p.acc_cols = acc_cols;

    const size_t b_bytes = (size_t)(Fi / kBK) * Fo * 128;
    const size_t fixed = 1024 + b_bytes + sizeof(Bars);
    const size_t max_smem = 227 * 1024;
    int stages = (int)((max_smem - fixed) / kStageBytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return GNN_ERR_UNSUPPORTED;
    p.stages = stages;
    const size_t smem = fixed + (size_t)stages * kStageBytes;

    const cudaError_t attr_err = func_attr(reinterpret_cast<const void *>(k_proj_tc),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (attr_err != cudaSuccess) return cuda_status(attr_err);
    const int64_t n_tiles = (n + kBM - 1) / kBM;
    const int grid = (int)std::min<int64_t>(n_tiles, sm_count());
    k_proj_tc<<<grid, kThreads, smem, s>>>(tm, p);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}


}  // namespace gnn
