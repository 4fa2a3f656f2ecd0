// gemm.cu -- NVFP4 block-scaled GEMM on the sm_103a tensor cores.
//
// D[m][n] = s_gA * s_gB * sum_k e2m1(a_mk) s_A(m, k/16) e2m1(b_nk) s_B(n, k/16),
// FP32 accumulation, BF16 or FP32 output: the Fprop / Dgrad / Wgrad GEMMs of
// an NVFP4 linear layer ("Full-Stack FP4", Sec. 2 Linear projection and
// Eq. (1)-(2); "Pretraining LLMs with NVFP4", Sec. 4 Mixed precision: FP4
// inputs, BF16/FP32 outputs).
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: per stage one 128x256-fp4 A box and one
//               256x256-fp4 B box (128-byte swizzle) plus the stage's block
//               scales (contiguous 512-byte groups of the tile layout) by
//               plain bulk copies, all completing on the stage's mbarrier;
//   warp 1      TMEM owner and MMA issuer: copies the stage's scales into
//               tensor memory (tcgen05.cp) and issues four
//               tcgen05.mma.kind::mxf4nvf4.block_scale (K = 64 each), then
//               commits the stage back to the producer;
//   warps 2-5   epilogue: drain the 128 x 256 FP32 accumulator from TMEM,
//               scale by s_gA * s_gB, convert and store.
// Every mbarrier wait is bounded (2 s); a wait that runs out sets the status
// word read by nvfp4_device_error and the CTA drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"
#include "kernels.h"

namespace nvfp4 {

static __device__ unsigned int g_gemm_status = 0;

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;                    // 256 fp4 per row per stage
constexpr int kStages = 4;
constexpr int kKStepsPerStage = 4;               // K = 64 per MMA
constexpr uint32_t kABytes = kBM * kBKBytes;     // 16 KiB
constexpr uint32_t kBBytes = kBN * kBKBytes;     // 32 KiB
constexpr uint32_t kSFABytes = kKStepsPerStage * 512;
constexpr uint32_t kSFBBytes = 2 * kKStepsPerStage * 512;
constexpr uint32_t kStageBytes = kABytes + kBBytes + kSFABytes + kSFBBytes;
constexpr int kNumEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kNumEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                   // 256 FP32 accumulator columns
constexpr uint32_t kSfCol0 = 256;                 // then the per-stage scale columns
constexpr uint32_t kSfColsPerStage = 4 * kKStepsPerStage + 8 * kKStepsPerStage;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

struct Params {
    uint32_t M, N;
    uint32_t m_tiles, n_tiles;
    uint32_t ksteps;           // ceil(K / 64): MMAs per tile, also 4-scale groups per row
    uint32_t kstages;          // ceil(ksteps / 4)
    uint32_t sfb_row_tiles;    // ceil(N / 128)
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* sga;
    const float* sgb;
    void* d;
    int64_t ldd;
    int out_fp32;
    int vec_store;             // every output row starts on a 16-byte boundary
};

// Instruction descriptor for kind::mxf4nvf4: A and B E2M1 (format 1) at bits
// 7 and 10, both K-major, N >> 3 at bit 17, UE4M3 scales (bit 23 = 0), M >> 7
// at bit 27, scale-factor ids 0.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 7) << 27);

__device__ __forceinline__ void record_timeout(volatile uint32_t* abort_flag) {
    *abort_flag = 1u;
    atomicOr(&g_gemm_status, kStatusTimeoutBit);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                     const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kNumEpiWarps);
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_barrier_init();
        prefetch_tmap(&tma_a);
        prefetch_tmap(&tma_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t num_tiles = p.m_tiles * p.n_tiles;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ producer
        uint32_t armed = 0, armed_parity = 0;   // per stage: copies issued, parity of their phase
        uint32_t stage = 0, phase = 0;
        for (uint32_t tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
            const uint32_t mt = tile % p.m_tiles, nt = tile / p.m_tiles;
            const bool b_hi = (2 * nt + 1) < p.sfb_row_tiles;
            for (uint32_t ks = 0; ks < p.kstages; ++ks) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, kTimeoutNs)) {
                    record_timeout(abort_flag);
                    break;
                }
                if (*abort_flag) break;
                const uint32_t k0 = ks * kKStepsPerStage;
                const uint32_t nk = min((uint32_t)kKStepsPerStage, p.ksteps - k0);
                const uint32_t bytes = kABytes + kBBytes + nk * 512u * (b_hi ? 3u : 2u);
                uint8_t* st = smem + stage * kStageBytes;
                mbar_arrive_expect_tx(&full[stage], bytes);
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                tma_load_2d(st, &tma_a, &full[stage], (int32_t)(ks * kBKBytes), (int32_t)(mt * kBM));
                tma_load_2d(st + kABytes, &tma_b, &full[stage], (int32_t)(ks * kBKBytes), (int32_t)(nt * kBN));
                bulk_load(st + kABytes + kBBytes, p.sfa + ((size_t)mt * p.ksteps + k0) * 512u, nk * 512u,
                          &full[stage]);
                bulk_load(st + kABytes + kBBytes + kSFABytes, p.sfb + ((size_t)(2 * nt) * p.ksteps + k0) * 512u,
                          nk * 512u, &full[stage]);
                if (b_hi)
                    bulk_load(st + kABytes + kBBytes + kSFABytes + kKStepsPerStage * 512u,
                              p.sfb + ((size_t)(2 * nt + 1) * p.ksteps + k0) * 512u, nk * 512u, &full[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // every copy this thread issued must land before the CTA exits
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            if ((armed >> s) & 1u) (void)mbar_wait(&full[s], (armed_parity >> s) & 1u, kTimeoutNs);
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------- MMA issuer
        uint32_t stage = 0, phase = 0, tiles_done = 0;
        for (uint32_t tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
            if (!mbar_wait(acc_empty, (tiles_done & 1u) ^ 1u, kTimeoutNs)) {
                record_timeout(abort_flag);
                break;
            }
            tc_fence_after();
            bool ok = true;
            for (uint32_t ks = 0; ks < p.kstages; ++ks) {
                if (!mbar_wait(&full[stage], phase, kTimeoutNs)) {
                    record_timeout(abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t nk = min((uint32_t)kKStepsPerStage, p.ksteps - ks * kKStepsPerStage);
                const uint32_t st = smem_u32(smem + stage * kStageBytes);
                const uint32_t sfa = st + kABytes + kBBytes, sfb = sfa + kSFABytes;
                const uint32_t sf_col = tmem + kSfCol0 + stage * kSfColsPerStage;
                for (uint32_t j = 0; j < nk; ++j) {
                    tmem_cp_32x128b_x4(sf_col + 4 * j, smem_desc(sfa + 512 * j, 0, 128, 0));
                    tmem_cp_32x128b_x4(sf_col + 16 + 8 * j, smem_desc(sfb + 512 * j, 0, 128, 0));
                    tmem_cp_32x128b_x4(sf_col + 16 + 8 * j + 4,
                                       smem_desc(sfb + kKStepsPerStage * 512 + 512 * j, 0, 128, 0));
                }
                for (uint32_t j = 0; j < nk; ++j) {
                    const uint64_t adesc = smem_desc(st + 32 * j, 16, 1024, 2);
                    const uint64_t bdesc = smem_desc(st + kABytes + 32 * j, 16, 1024, 2);
                    mma_nvf4(tmem + kAccCol, adesc, bdesc, kIdesc, sf_col + 4 * j, sf_col + 16 + 8 * j,
                             (ks | j) != 0 ? 1u : 0u);
                }
                tc_commit(&empty[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit(acc_full);
            ++tiles_done;
        }
        // all MMAs this thread issued complete before tensor memory is freed
        tc_commit(drain);
        (void)mbar_wait(drain, 0, kTimeoutNs);
    } else if (warp >= 2) {
        // ------------------------------------------------------- epilogue
        const uint32_t q = warp & 3u;   // TMEM lane quadrant this warp may access
        const float alpha = __fmul_rn(*p.sga, *p.sgb);
        uint32_t tiles_done = 0;
        for (uint32_t tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
            const uint32_t mt = tile % p.m_tiles, nt = tile / p.m_tiles;
            if (!mbar_wait(acc_full, tiles_done & 1u, kTimeoutNs)) {
                record_timeout(abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t row = mt * kBM + q * 32 + lane;
            const bool row_ok = row < p.M;
            for (uint32_t c = 0; c < kBN / 32; ++c) {
                const uint32_t n0 = nt * kBN + c * 32;
                if (n0 >= p.N) break;   // warp-uniform
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + ((q * 32u) << 16) + kAccCol + c * 32, v);
                tmem_ld_wait();
                if (!row_ok) continue;
                const bool full_chunk = p.vec_store && n0 + 32 <= p.N;
                if (p.out_fp32) {
                    float* dst = reinterpret_cast<float*>(p.d) + (int64_t)row * p.ldd + n0;
                    if (full_chunk) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            float4 o;
                            o.x = __fmul_rn(__uint_as_float(v[i + 0]), alpha);
                            o.y = __fmul_rn(__uint_as_float(v[i + 1]), alpha);
                            o.z = __fmul_rn(__uint_as_float(v[i + 2]), alpha);
                            o.w = __fmul_rn(__uint_as_float(v[i + 3]), alpha);
                            *reinterpret_cast<float4*>(dst + i) = o;
                        }
                    } else {
#pragma unroll
                        for (uint32_t i = 0; i < 32; ++i)
                            if (n0 + i < p.N) dst[i] = __fmul_rn(__uint_as_float(v[i]), alpha);
                    }
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.d) + (int64_t)row * p.ldd + n0;
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[2 * i]), alpha),
                                                                      __fmul_rn(__uint_as_float(v[2 * i + 1]), alpha));
                        packed[i] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                    if (full_chunk) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<uint4*>(dst + 2 * i) =
                                make_uint4(packed[i], packed[i + 1], packed[i + 2], packed[i + 3]);
                    } else {
#pragma unroll
                        for (uint32_t i = 0; i < 32; ++i)
                            if (n0 + i < p.N) dst[i] = (uint16_t)((packed[i / 2] >> (16 * (i & 1))) & 0xFFFFu);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            ++tiles_done;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host ---
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D map over packed codes: inner dimension K/2 bytes, outer `rows`.
bool make_codes_map(CUtensorMap* map, const GemmOperand& op, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(op.cols / 2), (cuuint64_t)op.rows};
    const cuuint64_t strides[1] = {(cuuint64_t)op.ld_codes};
    const cuuint32_t box[2] = {(cuuint32_t)kBKBytes, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(op.codes), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int device_sm_count() {
    static int counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (counts[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        counts[dev] = n > 0 ? n : 1;
    }
    return counts[dev];
}

cudaError_t launch_gemm(const GemmOperand& a, const GemmOperand& b, void* d, int64_t ldd, bool out_fp32,
                        cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_codes_map(&ma, a, kBM) || !make_codes_map(&mb, b, kBN)) return cudaErrorInvalidValue;
    static bool attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    Params p{};
    p.M = (uint32_t)a.rows;
    p.N = (uint32_t)b.rows;
    p.m_tiles = (uint32_t)((a.rows + kBM - 1) / kBM);
    p.n_tiles = (uint32_t)((b.rows + kBN - 1) / kBN);
    p.ksteps = (uint32_t)((a.cols + 63) / 64);
    p.kstages = (p.ksteps + kKStepsPerStage - 1) / kKStepsPerStage;
    p.sfb_row_tiles = (uint32_t)((b.rows + 127) / 128);
    p.sfa = a.scales;
    p.sfb = b.scales;
    p.sga = a.sg;
    p.sgb = b.sg;
    p.d = d;
    p.ldd = ldd;
    p.out_fp32 = out_fp32 ? 1 : 0;
    const int64_t esz = out_fp32 ? 4 : 2;
    p.vec_store = ((reinterpret_cast<uintptr_t>(d) & 15u) == 0 && (ldd * esz) % 16 == 0) ? 1 : 0;
    const uint32_t tiles = p.m_tiles * p.n_tiles;
    const uint32_t sms = (uint32_t)device_sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    gemm_nvf4_kernel<<<grid, kThreads, kSmemBytes, stream>>>(ma, mb, p);
    return cudaGetLastError();
}

cudaError_t gemm_read_and_clear_status(unsigned int* status) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) e = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof zero);
    *status = v;
    return e;
}

}  // namespace nvfp4
