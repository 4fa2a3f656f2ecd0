// gemm.cu -- NVFP4 block-scaled GEMM on the sm_103a tensor cores.
//
// D[m][n] = s_gA * s_gB * sum_k e2m1(a_mk) s_A(m, k/16) e2m1(b_nk) s_B(n, k/16),
// FP32 accumulation, BF16 or FP32 output: the Fprop / Dgrad / Wgrad GEMMs of
// an NVFP4 linear layer ("Full-Stack FP4", Sec. 2 Linear projection and
// Eq. (1)-(2); "Pretraining LLMs with NVFP4", Sec. 4 Mixed precision: FP4
// inputs, BF16/FP32 outputs).
//
// Design: CTA pairs (clusters of 2, one CTA per SM), persistent over 256 x 256
// output tiles.  The pair's tile is computed by tcgen05.mma.cta_group::2: each
// CTA holds 128 rows of A and 128 of the 256 B rows in its shared memory and
// 128 accumulator rows in its tensor memory, so each SM streams half of B.
// Per CTA (16 warps):
//   warps 0, 2  TMA producers, one copy per stage each: the 128-row A box and
//               the 128-row B box (256 fp4 of K, 128-byte swizzle), both
//               completing on the leader CTA's full barrier;
//   warp 3      scale producer: the stage's block scales (this CTA's 128 A
//               rows, all 256 B rows) as two 3-D TMA boxes of the tile layout
//               onto a local barrier;
//   warp 1      TMEM allocation for the pair; in the leader CTA, the MMA
//               issuer: one barrier wait, four block-scaled MMAs (K = 64 each)
//               and one commit per stage, nothing else (the tensor pipe only
//               stays busy while the issuing thread keeps up with it);
//   warps 4-7   scale warps, one per TMEM lane quadrant: move the stage's
//               scales from shared memory into the stage's TMEM columns with
//               tcgen05.st (off the MMA pipe) and arrive on the leader's full
//               barrier, which therefore completes when both CTAs' tiles have
//               landed and all eight scale warps are done;
//   warps 8-15  epilogue, two per lane quadrant (one per 128-column half):
//               load the warp's 128 accumulator columns into registers under
//               one wait, release the accumulator to the leader, scale by
//               s_gA * s_gB, stage the results in 128-byte-swizzled shared
//               memory and write them with TMA stores (unaligned outputs:
//               direct stores).
// The warp groups split the register file with setmaxnreg (64 / 72 / 184 x2
// per thread) so that the epilogue holds a whole accumulator half.
// Every mbarrier wait is bounded (2 s); a wait that runs out sets the status
// word read by nvfp4_device_error and both CTAs drain and exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "bounds.cuh"
#include "device_common.cuh"
#include "kernels.h"

namespace nvfp4 {

static __device__ unsigned int g_gemm_status = 0;

// Wait limit of the next GEMM launch that withholds one arrival (0: none
// armed); set by arm_gemm_fault, consumed by launch_gemm.
static std::atomic<uint64_t> g_armed_fault_ns{0};

namespace {

constexpr int kNumEpiWarpsStaging = 8;
constexpr int kPairM = 256;                      // output rows per CTA pair
constexpr int kCtaM = 128;                       // rows of A (and accumulator lanes) per CTA
constexpr int kBN = 256;                         // output columns per tile
constexpr int kCtaN = 128;                       // rows of B per CTA
constexpr int kBKBytes = 128;                    // 256 fp4 of K per row per stage
constexpr int kStages = 5;
constexpr int kKStepsPerStage = 4;               // K = 64 per MMA
constexpr uint32_t kABytes = kCtaM * kBKBytes;   // 16 KiB
constexpr uint32_t kBBytes = kCtaN * kBKBytes;   // 16 KiB
constexpr uint32_t kSFABytes = kKStepsPerStage * 512;
constexpr uint32_t kSFBBytes = 2 * kKStepsPerStage * 512;
constexpr uint32_t kStageBytes = kABytes + kBBytes + kSFABytes + kSFBBytes;
constexpr uint32_t kStagingBytes = kNumEpiWarpsStaging * 4096;   // 32 rows x 64 BF16 columns per epilogue warp
constexpr int kProdAWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kProdBWarp = 2;
constexpr int kProdSfWarp = 3;
constexpr int kFirstSfWarp = 4;
constexpr int kNumSfWarps = 4;
constexpr int kFirstEpiWarp = kFirstSfWarp + kNumSfWarps;
constexpr int kNumEpiWarps = 8;
constexpr int kThreads = 32 * (kFirstEpiWarp + kNumEpiWarps);
// the leader's full barrier: its A producer's arrive.expect_tx plus the scale
// warps of both CTAs
constexpr uint32_t kFullArrivals = 1 + 2 * kNumSfWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                   // 256 FP32 accumulator columns
constexpr uint32_t kSfCol0 = 256;                 // then the per-stage scale columns
constexpr uint32_t kSfColsPerStage = 4 * kKStepsPerStage + 8 * kKStepsPerStage;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + kStagingBytes + 1024 /*align*/ + 256 /*barriers*/;

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
    uint32_t M, N;
    uint32_t m_tiles, n_tiles;   // 256-row and 256-column tiles
    uint32_t ksteps;             // ceil(K / 64): MMAs per tile, also 4-scale groups per row
    uint32_t kstages;            // ceil(ksteps / 4)
    uint32_t last_nk;            // MMAs in a tile's last stage (1..4)
    const float* sga;
    const float* sgb;
    void* d;
    int64_t ldd;
    int out_fp32;
    int vec_store;               // every output row starts on a 16-byte boundary
    int tma_store;               // output written through the D tensor map (BF16 or FP32)
    uint32_t n_tma;              // columns the D map covers: N cut to whole 16-byte pieces
    int n_fast;                  // tile order: N tiles vary fastest (else M tiles)
    uint32_t lora_stages;        // 64-deep BF16 stages of the low-rank term per tile (0: none)
    float* amax_out;             // [2]: max |D| and max |RHT along D's rows| (BF16 TMA path), or null
    uint32_t rht_sgn[16];        // the RHT mask's sign flips as XOR words on packed bf16 pairs (row i: bit i)
    float alpha;                 // extra factor on the product (1 for a plain GEMM)
    const void* c;               // D = alpha s_gA s_gB A B^T + beta C: C [M][ldc] of D's dtype, or null
    int64_t ldc;
    float beta;
    int c_vec;                   // every row of C starts on a 16-byte boundary
    int c_staged;                // C copied into the epilogue's slices by the lanes (cp.async)
    uint64_t timeout_ns;         // limit of every mbarrier wait
    uint32_t withhold;           // test support: the leader's first scale-warp arrival is left out
    Extent xd;                   // the bytes of D the epilogue's direct stores may write
};

// 32 consecutive values of C's row `row` from column n0 (zeros past M or N):
// BF16 as 16 packed pairs, FP32 as 32 floats.
__device__ __forceinline__ void load_c_bf16x32(const Params& p, uint32_t row, uint32_t n0, uint32_t* w) {
    const uint16_t* src = static_cast<const uint16_t*>(p.c) + (int64_t)row * p.ldc + n0;
    if (row < p.M && p.c_vec && n0 + 32 <= p.N) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 u = *reinterpret_cast<const uint4*>(src + 8 * j);
            w[4 * j] = u.x;
            w[4 * j + 1] = u.y;
            w[4 * j + 2] = u.z;
            w[4 * j + 3] = u.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t lo = (row < p.M && n0 + 2 * i < p.N) ? src[2 * i] : 0u;
            const uint32_t hi = (row < p.M && n0 + 2 * i + 1 < p.N) ? src[2 * i + 1] : 0u;
            w[i] = lo | (hi << 16);
        }
    }
}
__device__ __forceinline__ void load_c_f32x32(const Params& p, uint32_t row, uint32_t n0, float* f) {
    const float* src = static_cast<const float*>(p.c) + (int64_t)row * p.ldc + n0;
    if (row < p.M && p.c_vec && n0 + 32 <= p.N) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 u = *reinterpret_cast<const float4*>(src + 4 * j);
            f[4 * j] = u.x;
            f[4 * j + 1] = u.y;
            f[4 * j + 2] = u.z;
            f[4 * j + 3] = u.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = (row < p.M && n0 + i < p.N) ? src[i] : 0.0f;
    }
}

// L2 prefetch of the C values one epilogue lane combines for a tile: its
// row's 128 columns from n0 (BF16: 256 bytes, FP32: 512 bytes), in 128-byte
// lines, only inside C.  Issued before the lane waits for the tile's
// accumulator, so that C's reads after it hit L2 instead of waiting on DRAM.
__device__ __forceinline__ void prefetch_c_row(const Params& p, uint32_t row, uint32_t n0) {
    if (row >= p.M || n0 >= p.N) return;
    const int64_t esz = p.out_fp32 ? 4 : 2;
    const char* base = static_cast<const char*>(p.c) + ((int64_t)row * p.ldc + n0) * esz;
    const uint32_t cols = (p.N - n0) < 128u ? (p.N - n0) : 128u;
    const int64_t bytes = (int64_t)cols * esz;
    for (int64_t off = 0; off < bytes; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(base + off));
}

// One round's 32 rows x 128 bytes of C at column x, row y into an epilogue
// warp's slice (128-byte swizzle, as the output's TMA store reads it), by
// the lanes' own asynchronous copies: instruction i moves rows 4i .. 4i+3,
// eight 16-byte pieces each; pieces past N and rows past M read as zero.
// The copies go through the load/store path, not through the TMA unit that
// carries the operand ring.  Completed by cp_async_wait_all.
__device__ __forceinline__ void load_c_slice_async(const Params& p, uint8_t* slice, uint32_t lane, uint32_t x,
                                                   uint32_t y) {
    const uint32_t esz = p.out_fp32 ? 4u : 2u;
    const uint32_t per = 16u / esz;   // columns per piece
    const uint32_t ch = lane & 7u;
    const uint32_t c0 = x + ch * per;
    const uint32_t nbytes = c0 >= p.N ? 0u : ((p.N - c0) >= per ? 16u : (p.N - c0) * esz);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t rr = 4u * (uint32_t)i + (lane >> 3);
        const uint32_t grow = y + rr;
        const uint32_t n = grow < p.M ? nbytes : 0u;
        const char* src = static_cast<const char*>(p.c) + (n ? ((int64_t)grow * p.ldc + c0) * esz : 0);
        const uint32_t dst = smem_u32(slice + rr * 128u + ((ch ^ (rr & 7u)) * 16u));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// One output value: RN(acc * alpha) + RN(beta * c) in binary32 (the C term
// only when the call has one).
__device__ __forceinline__ float epi_value(uint32_t acc_bits, float alpha, bool has_c, float beta, float c) {
    const float y = __fmul_rn(__uint_as_float(acc_bits), alpha);
    return has_c ? __fadd_rn(y, __fmul_rn(beta, c)) : y;
}

// Output tile of a linear tile index.  Tiles that run at the same time share
// the slow index, so its operand block is read from DRAM once and served from
// L2 to every pair; the fast index cycles through the whole other operand,
// which the host chooses to be the smaller one so that it stays in L2.
__device__ __forceinline__ void tile_coords(uint32_t tile, const Params& p, uint32_t& mt, uint32_t& nt) {
    if (p.n_fast) {
        nt = tile % p.n_tiles;
        mt = tile / p.n_tiles;
    } else {
        mt = tile % p.m_tiles;
        nt = tile / p.m_tiles;
    }
}

// Instruction descriptor for kind::mxf4nvf4: A and B E2M1 (format 1) at bits
// 7 and 10, both K-major, N >> 3 at bit 17, UE4M3 scales (bit 23 = 0), M >> 7
// at bit 27 (M = 256 for the pair), scale-factor ids 0.
constexpr uint32_t kIdesc =
    (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kPairM >> 7) << 27);

// Instruction descriptor for kind::f16 (the low-rank term): FP32 D (bit 4),
// A and B BF16 (format 1 at bits 7 and 10), both K-major, N >> 3 at bit 17,
// M >> 4 at bit 24 (M = 256 for the pair).
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                                ((uint32_t)(kPairM >> 4) << 24);

// Four pair MMAs of kind::f16 over one 64-deep BF16 stage (16 per MMA; the
// descriptors advance by 32 bytes like the FP4 steps); accumulates onto D
// unless the stage is the first MMA work of the tile.
__device__ __forceinline__ void mma_bf16_pair_stage(uint32_t d_tmem, uint32_t a_lo, uint32_t desc_hi,
                                                    uint32_t b_off, uint32_t accumulate_first) {
    asm volatile(
        "{\n\t"
        ".reg .b32 a1, a2, a3, b0, b1, b2, b3;\n\t"
        ".reg .b64 da0, da1, da2, da3, db0, db1, db2, db3;\n\t"
        ".reg .pred p;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "add.u32 a1, %1, 2;\n\tadd.u32 a2, %1, 4;\n\tadd.u32 a3, %1, 6;\n\t"
        "add.u32 b0, %1, %4;\n\tadd.u32 b1, b0, 2;\n\tadd.u32 b2, b0, 4;\n\tadd.u32 b3, b0, 6;\n\t"
        "mov.b64 da0, {%1, %2};\n\tmov.b64 da1, {a1, %2};\n\tmov.b64 da2, {a2, %2};\n\tmov.b64 da3, {a3, %2};\n\t"
        "mov.b64 db0, {b0, %2};\n\tmov.b64 db1, {b1, %2};\n\tmov.b64 db2, {b2, %2};\n\tmov.b64 db3, {b3, %2};\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da0, db0, %5, p;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da1, db1, %5, 1;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da2, db2, %5, 1;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], da3, db3, %5, 1;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_lo), "r"(desc_hi), "r"(accumulate_first), "r"(b_off), "n"(kIdescBf16)
        : "memory");
}

__device__ __forceinline__ void record_timeout(volatile uint32_t* abort_flag) {
    *abort_flag = 1u;
    atomicOr(&g_gemm_status, kStatusTimeoutBit);
}

// Named barrier over the scale warps (id 2); id 0 and the cluster barrier
// are used elsewhere.
__device__ __forceinline__ void scale_bar() {
    asm volatile("bar.sync 2, %0;" ::"n"(32 * kNumSfWarps) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Packed binary32 pairs (two columns in one 64-bit register pair): each lane
// of an add.f32x2 / sub.f32x2 rounds like the scalar operation.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void f32x2_butterfly(uint64_t& a, uint64_t& b) {
    uint64_t s, d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(a), "l"(b));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    a = s;
    b = d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// The amax contributions of one 32-row x 64-column BF16 slice of the output
// (128-byte swizzled, row j at j * 128 bytes): lane c takes columns 2c and
// 2c + 1 down the 32 rows, i.e. two 16-row blocks per column, and folds in
// max |x| and max |H16 D x| of each block, the transform in the quantizer's
// order (signs, then butterfly stages 0..3 as (a + b, a - b)), both columns
// at once in packed pairs; the 1/4 is applied to the final maximum, exactly.
__device__ __forceinline__ void slice_amax(const uint8_t* slice, uint32_t lane, const Params& p,
                                           float& amax_plain, float& amax_rht) {
    const uint32_t chunk = lane >> 2, word = (lane & 3u) * 4u;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint64_t t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t j = 16u * blk + i;
            uint32_t w = *reinterpret_cast<const uint32_t*>(slice + j * 128u + ((chunk ^ (j & 7u)) << 4) + word);
            w ^= p.rht_sgn[i];     // D: both columns' sign bits
            const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
            amax_plain = fmax3(amax_plain, fabsf(lo), fabsf(hi));
            t[i] = f32x2_pack(lo, hi);
        }
#pragma unroll
        for (int st = 0; st < 4; ++st) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (!(i & (1 << st))) f32x2_butterfly(t[i], t[i | (1 << st)]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float lo, hi;
            f32x2_unpack(t[i], lo, hi);
            amax_rht = fmax3(amax_rht, fabsf(lo), fabsf(hi));
        }
    }
}

// The columns [max(x, n_tma), min(x + cols, N)) of this lane's row of a
// staged round (x: the round's first column, cols its width; the slice holds
// the round's 32 rows, row = lane, 128-byte swizzled).  A TMA store writes
// whole 16-byte pieces of a row even past the tensor map's last column, so
// the D map ends at n_tma, the last 16-byte boundary at or below N, and the
// lanes store the at most 7 (BF16) or 3 (FP32) columns after it themselves.
__device__ __forceinline__ void store_round_tail(const Params& p, const uint8_t* slice, uint32_t lane,
                                                 uint32_t row, uint32_t x, uint32_t cols) {
    const uint32_t lo = x > p.n_tma ? x : p.n_tma, hi = x + cols < p.N ? x + cols : p.N;
    if (row >= p.M || lo >= hi) return;
    const uint32_t esz = p.out_fp32 ? 4u : 2u;
    for (uint32_t c = lo; c < hi; ++c) {
        const uint32_t b = (c - x) * esz;
        const uint8_t* src = slice + lane * 128u + (((b >> 4) ^ (lane & 7u)) << 4) + (b & 15u);
        if (p.out_fp32)
            store_out(reinterpret_cast<float*>(p.d) + (int64_t)row * p.ldd + c, *reinterpret_cast<const float*>(src),
                      p.xd);
        else
            store_out(reinterpret_cast<uint16_t*>(p.d) + (int64_t)row * p.ldd + c,
                      *reinterpret_cast<const uint16_t*>(src), p.xd);
    }
}

// Epilogue variants: the plain product; the product plus the output's two
// tensor amaxes (p.amax_out); alpha times the product plus beta C (p.c).
enum EpiMode { kEpiPlain = 0, kEpiAmax = 1, kEpiC = 2 };

template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                     const __grid_constant__ CUtensorMap tma_sfa, const __grid_constant__ CUtensorMap tma_sfb,
                     const __grid_constant__ CUtensorMap tma_d, const __grid_constant__ CUtensorMap tma_u,
                     const __grid_constant__ CUtensorMap tma_v, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + kStages * kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(staging + kStagingBytes);   // leader: tiles + scale warps
    uint64_t* sf_full = full + kStages;          // local: this CTA's scale bytes
    uint64_t* empty = sf_full + kStages;         // local: released by the leader's commit
    uint64_t* acc_full = empty + kStages;        // local: released by the leader's commit
    uint64_t* acc_empty = acc_full + 1;          // leader: 2 x kNumEpiWarps arrivals
    uint64_t* drain = acc_empty + 1;             // leader
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    volatile uint32_t* sf_ok = tmem_slot + 4;    // [2]: scales-landed verdicts, by stage-count parity

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kFullArrivals);
            mbar_init(&sf_full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kNumEpiWarps);
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == kProdAWarp && lane == 0) {
        prefetch_tmap(&tma_a);
        if (p.lora_stages) prefetch_tmap(&tma_u);
    }
    if (warp == kProdBWarp && lane == 0) {
        prefetch_tmap(&tma_b);
        if (p.lora_stages) prefetch_tmap(&tma_v);
    }
    if (warp == kProdSfWarp && lane == 0) {
        prefetch_tmap(&tma_sfa);
        prefetch_tmap(&tma_sfb);
    }
    if (warp == kFirstEpiWarp && lane == 0 && p.tma_store) prefetch_tmap(&tma_d);
    if (warp == kMmaWarp) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t num_tiles = p.m_tiles * p.n_tiles;
    const uint32_t first_tile = cluster_id_x(), tile_stride = num_clusters_x();

    // Registers per thread by warp group (setmaxnreg): producers and MMA
    // issuer 64, scale warps 72, epilogue 184, so that each epilogue warp
    // holds its whole 128-column accumulator half in registers and hands the
    // accumulator back after one wait.  The launch gives all 512 threads 128
    // (checked on the host): 128 * (64 + 72) + 256 * 184 = 64512 <= 65536.
    if (warp < (uint32_t)kFirstSfWarp) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
        if (warp != (uint32_t)kMmaWarp) {
            if (lane == 0) {
                // ------------------------------------------------- producers
                // Three warps, one or two copies each per stage: a single thread
                // cannot issue a stage's five copies fast enough.
                uint32_t armed = 0, armed_parity = 0;   // per stage: copies issued, parity of their phase
                uint32_t stage = 0, phase = 0;
                const uint32_t leader_full0 = map_to_cta(smem_u32(full), 0);
                for (uint32_t tile = first_tile; tile < num_tiles && !*abort_flag; tile += tile_stride) {
                    uint32_t mt, nt;
                    tile_coords(tile, p, mt, nt);
                    for (uint32_t ks = 0; ks < p.kstages; ++ks) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns)) {
                            record_timeout(abort_flag);
                            break;
                        }
                        if (*abort_flag) break;
                        uint8_t* st = smem + stage * kStageBytes;
                        const uint32_t leader_full = leader_full0 + stage * 8u;
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        if (warp == kProdAWarp) {
                            if (leader) mbar_arrive_expect_tx(&full[stage], 2u * (kABytes + kBBytes));
                            tma_load_2d_pair(st, &tma_a, leader_full, (int32_t)(ks * kBKBytes),
                                             (int32_t)(mt * kPairM + rank * kCtaM));
                        } else if (warp == kProdBWarp) {
                            tma_load_2d_pair(st + kABytes, &tma_b, leader_full, (int32_t)(ks * kBKBytes),
                                             (int32_t)(nt * kBN + rank * kCtaN));
                        } else {
                            // scale boxes: 4 groups of 512 bytes per 128-row tile;
                            // groups past K and row tiles past M / N read as zero
                            uint8_t* sfa_s = st + kABytes + kBBytes;
                            mbar_arrive_expect_tx(&sf_full[stage], kSFABytes + kSFBBytes);
                            tma_load_3d(sfa_s, &tma_sfa, &sf_full[stage], 0, (int32_t)(ks * kKStepsPerStage),
                                        (int32_t)(2 * mt + rank));
                            tma_load_3d(sfa_s + kSFABytes, &tma_sfb, &sf_full[stage], 0,
                                        (int32_t)(ks * kKStepsPerStage), (int32_t)(2 * nt));
                        }
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    // the low-rank term: 64 BF16 columns of U' and V per stage in
                    // the A and B slots (the same 16 KiB boxes), no scales
                    for (uint32_t ls = 0; ls < p.lora_stages && !*abort_flag; ++ls) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns)) {
                            record_timeout(abort_flag);
                            break;
                        }
                        uint8_t* st = smem + stage * kStageBytes;
                        const uint32_t leader_full = leader_full0 + stage * 8u;
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        if (warp == kProdAWarp) {
                            if (leader) mbar_arrive_expect_tx(&full[stage], 2u * (kABytes + kBBytes));
                            tma_load_2d_pair(st, &tma_u, leader_full, (int32_t)(ls * 64u),
                                             (int32_t)(mt * kPairM + rank * kCtaM));
                        } else if (warp == kProdBWarp) {
                            tma_load_2d_pair(st + kABytes, &tma_v, leader_full, (int32_t)(ls * 64u),
                                             (int32_t)(nt * kBN + rank * kCtaN));
                        } else {
                            mbar_arrive(&sf_full[stage]);
                        }
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                // every copy must land before the pair exits: the leader's full
                // barriers count both CTAs' tile bytes, sf_full this CTA's scales
    #pragma unroll
                for (int s = 0; s < kStages; ++s) {
                    if (!((armed >> s) & 1u)) continue;
                    const uint32_t par = (armed_parity >> s) & 1u;
                    if (warp == kProdAWarp && leader) (void)mbar_wait_cluster(&full[s], par, p.timeout_ns);
                    if (warp == kProdSfWarp) (void)mbar_wait(&sf_full[s], par, p.timeout_ns);
                }
            }
        } else {
            if (leader && lane == 0) {
                // ------------------------------------------------ MMA issuer
                // The tensor pipe only stays busy while this thread keeps up with
                // it, so the loop body is one barrier wait, the stage's four MMAs
                // (one asm block, descriptors built from 32-bit low words) and one
                // commit, with every stage address advanced by an add.  (Splitting
                // the four MMAs to wait for the next stage in between measured
                // slower.)
                constexpr uint32_t kStageDesc = kStageBytes >> 4;   // descriptor address units
                constexpr uint32_t kBOff = kABytes >> 4;
                const uint64_t desc0 = smem_desc(smem_u32(smem), 16, 1024, 2);
                const uint32_t lo0 = (uint32_t)desc0, hi = (uint32_t)(desc0 >> 32);
                const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
                const uint32_t sfc0 = tmem + kSfCol0;
                const uint32_t acc = tmem + kAccCol;
                const uint32_t kst = p.kstages;
                const bool tail = p.last_nk != (uint32_t)kKStepsPerStage;
                uint32_t stage = 0, phase = 0, tiles_done = 0;
                uint32_t alo = lo0, sfc = sfc0, fa = full0, ea = empty0;
                for (uint32_t tile = first_tile; tile < num_tiles && !*abort_flag; tile += tile_stride) {
                    if (!mbar_wait_cluster(acc_empty, (tiles_done & 1u) ^ 1u, p.timeout_ns)) {
                        record_timeout(abort_flag);
                        break;
                    }
                    tc_fence_after();
                    bool ok = true;
                    for (uint32_t ks = 0; ks < kst; ++ks) {
                        if (!mbar_wait_addr(fa, phase, p.timeout_ns)) {
                            record_timeout(abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (ks != 0 && (ks + 1u != kst || !tail)) {
                            mma_nvf4_pair_stage<true, kBOff>(acc, alo, hi, kIdesc, sfc);
                        } else if (ks + 1u != kst || !tail) {
                            mma_nvf4_pair_stage<false, kBOff>(acc, alo, hi, kIdesc, sfc);
                        } else {
                            // last stage of a K that is not a multiple of 256
                            const uint64_t da = ((uint64_t)hi << 32) | alo;
                            for (uint32_t j = 0; j < p.last_nk; ++j)
                                mma_nvf4_pair(acc, da + 2 * j, da + kBOff + 2 * j, kIdesc, sfc + 4 * j,
                                              sfc + 16 + 8 * j, (ks | j) != 0 ? 1u : 0u);
                        }
                        tc_commit_pair_multicast_addr(ea, 0x3);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                            alo = lo0;
                            sfc = sfc0;
                            fa = full0;
                            ea = empty0;
                        } else {
                            alo += kStageDesc;
                            sfc += kSfColsPerStage;
                            fa += 8u;
                            ea += 8u;
                        }
                    }
                    for (uint32_t ls = 0; ok && ls < p.lora_stages; ++ls) {
                        if (!mbar_wait_addr(fa, phase, p.timeout_ns)) {
                            record_timeout(abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        mma_bf16_pair_stage(acc, alo, hi, kBOff, (kst | ls) != 0 ? 1u : 0u);
                        tc_commit_pair_multicast_addr(ea, 0x3);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                            alo = lo0;
                            sfc = sfc0;
                            fa = full0;
                            ea = empty0;
                        } else {
                            alo += kStageDesc;
                            sfc += kSfColsPerStage;
                            fa += 8u;
                            ea += 8u;
                        }
                    }
                    if (!ok) break;
                    tc_commit_pair_multicast(acc_full, 0x3);
                    ++tiles_done;
                }
                // all MMAs complete before either CTA frees its tensor memory
                tc_commit_pair_multicast(drain, 0x1);
                (void)mbar_wait(drain, 0, p.timeout_ns);
            }
        }
    } else if (warp < (uint32_t)kFirstEpiWarp) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
        // ------------------------------------------------------ scale warps
        // Lane i of quadrant q holds, per K = 64 step j, 4 columns of A scales
        // (bytes 16i.. of the step's 512-byte group: rows i, i+32, i+64, i+96)
        // and 8 columns of B scales (both 128-row halves of the N tile).
        const uint32_t q = warp & 3u;
        const uint32_t leader_full0 = map_to_cta(smem_u32(full), 0);
        uint32_t stage = 0, phase = 0, count = 0;
        for (uint32_t tile = first_tile; tile < num_tiles; tile += tile_stride) {
            bool ok = true;
            for (uint32_t ks = 0; ks < p.kstages; ++ks, ++count) {
                // one thread waits, the other scale warps sleep in a named
                // barrier; all leave together
                if (warp == (uint32_t)kFirstSfWarp && lane == 0) {
                    bool landed = !*abort_flag && mbar_wait(&sf_full[stage], phase, p.timeout_ns);
                    if (!landed && !*abort_flag) record_timeout(abort_flag);
                    sf_ok[count & 1u] = landed ? 1u : 0u;
                }
                __syncwarp();
                scale_bar();
                if (!sf_ok[count & 1u]) {
                    ok = false;
                    break;
                }
                const uint8_t* sfa = smem + stage * kStageBytes + kABytes + kBBytes;
                const uint8_t* sfb = sfa + kSFABytes;
                uint32_t ra[16], rb[32];
#pragma unroll
                for (int j = 0; j < kKStepsPerStage; ++j) {
                    const uint4 w = *reinterpret_cast<const uint4*>(sfa + 512 * j + 16 * lane);
                    ra[4 * j + 0] = w.x;
                    ra[4 * j + 1] = w.y;
                    ra[4 * j + 2] = w.z;
                    ra[4 * j + 3] = w.w;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 u =
                            *reinterpret_cast<const uint4*>(sfb + kKStepsPerStage * 512 * h + 512 * j + 16 * lane);
                        rb[8 * j + 4 * h + 0] = u.x;
                        rb[8 * j + 4 * h + 1] = u.y;
                        rb[8 * j + 4 * h + 2] = u.z;
                        rb[8 * j + 4 * h + 3] = u.w;
                    }
                }
                const uint32_t col = tmem + ((q * 32u) << 16) + kSfCol0 + stage * kSfColsPerStage;
                tmem_st_32x32b_x16(col, ra);
                tmem_st_32x32b_x32(col + 16, rb);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                // (test support: with p.withhold the leader's first scale warp
                // never arrives for the first stage, so the MMA issuer's wait
                // on that full barrier runs out)
                if (lane == 0 && !(p.withhold && count == 0 && leader && warp == (uint32_t)kFirstSfWarp))
                    mbar_arrive_cluster(leader_full0 + stage * 8u);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // low-rank stages carry no scales: only the arrival on full
            for (uint32_t ls = 0; ok && ls < p.lora_stages; ++ls, ++count) {
                if (warp == (uint32_t)kFirstSfWarp && lane == 0) {
                    bool landed = !*abort_flag && mbar_wait(&sf_full[stage], phase, p.timeout_ns);
                    if (!landed && !*abort_flag) record_timeout(abort_flag);
                    sf_ok[count & 1u] = landed ? 1u : 0u;
                }
                __syncwarp();
                scale_bar();
                if (!sf_ok[count & 1u]) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_cluster(leader_full0 + stage * 8u);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 184;" ::: "memory");
        // --------------------------------------------------------- epilogue
        const uint32_t q = warp & 3u;                          // TMEM lane quadrant
        const uint32_t half = (warp - kFirstEpiWarp) >> 2;     // 128-column half of the tile
        const float alpha = __fmul_rn(__fmul_rn(*p.sga, *p.sgb), p.alpha);
        constexpr bool kAmax = kMode == kEpiAmax;
        constexpr bool has_c = kMode == kEpiC;
        const uint32_t leader_acc_empty = map_to_cta(smem_u32(acc_empty), 0);
        // amax of the BF16 output for its quantization (rows of one warp are
        // lanes, so a 16-row block of a column is 16 lanes): the plain max
        // and the max after the RHT along the rows (sign of this lane's row,
        // then butterfly stages by shuffles; stage s: lanes with bit s set
        // take partner - t, the others t + partner)
        float amax_plain = 0.0f, amax_rht = 0.0f;
        const uint32_t row_local = q * 32 + lane;
        uint32_t tiles_done = 0;
        for (uint32_t tile = first_tile; tile < num_tiles; tile += tile_stride) {
            uint32_t mt, nt;
            tile_coords(tile, p, mt, nt);
            if constexpr (has_c)
                prefetch_c_row(p, mt * kPairM + rank * kCtaM + row_local, nt * kBN + half * 128);
            // One thread per warp waits for the accumulator, suspended in the
            // barrier's try_wait (no issue slots taken from the MMA issuer);
            // each warp wakes on the barrier itself, not behind a named
            // barrier that a single waiter would have to open (about 500
            // cycles per tile).
            uint32_t ready = 0;
            if (lane == 0) {
                ready = (!*abort_flag && mbar_wait_cluster(acc_full, tiles_done & 1u, p.timeout_ns)) ? 1u : 0u;
                if (!ready && !*abort_flag) record_timeout(abort_flag);
            }
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t row0 = mt * kPairM + rank * kCtaM;   // first row of this CTA's half
            const uint32_t row = row0 + row_local;
            const uint32_t nbase = nt * kBN + half * 128;
            const uint32_t taddr = tmem + ((q * 32u) << 16) + kAccCol + half * 128;
            if (has_c && p.c_staged) {
                // C through this warp's 4 KiB slice: each round the lanes copy
                // the round's 32 rows of C into the slice (the output map's
                // box and swizzle), every lane replaces its row's values by
                // the outputs in place, and the slice goes out with a TMA
                // store.  BF16: two rounds of 64 columns; FP32: four of 32.
                uint8_t* slice = staging + (half * 4 + q) * 4096u;
                uint32_t v[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, v[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(leader_acc_empty);
                const uint32_t y = row0 + q * 32;
                const int rounds = p.out_fp32 ? 4 : 2;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r >= rounds) break;
                    const uint32_t x = nbase + (uint32_t)r * (p.out_fp32 ? 32u : 64u);
                    // the slice's previous store must have read it before C lands in it
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    load_c_slice_async(p, slice, lane, x, y);
                    // each lane waits for its own copies; the warp barrier then
                    // makes every lane's pieces visible to the others
                    cp_async_wait_all();
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint4* cell = reinterpret_cast<uint4*>(slice + lane * 128u + ((uint32_t)i ^ (lane & 7u)) * 16u);
                        const uint4 cw = *cell;
                        uint4 o;
                        if (p.out_fp32) {
                            // columns 4i .. 4i+3 of round r = chunk r
                            o.x = __float_as_uint(epi_value(v[r][4 * i], alpha, true, p.beta, __uint_as_float(cw.x)));
                            o.y = __float_as_uint(epi_value(v[r][4 * i + 1], alpha, true, p.beta, __uint_as_float(cw.y)));
                            o.z = __float_as_uint(epi_value(v[r][4 * i + 2], alpha, true, p.beta, __uint_as_float(cw.z)));
                            o.w = __float_as_uint(epi_value(v[r][4 * i + 3], alpha, true, p.beta, __uint_as_float(cw.w)));
                        } else {
                            // columns 8i .. 8i+7 of round r = chunk 2r + i/4, from 8 (i % 4)
                            const uint32_t* a = &v[2 * r + (i >> 2)][8 * (i & 3)];
                            o.x = pack_bf16x2(epi_value(a[0], alpha, true, p.beta, bf16lo(cw.x)),
                                              epi_value(a[1], alpha, true, p.beta, bf16hi(cw.x)));
                            o.y = pack_bf16x2(epi_value(a[2], alpha, true, p.beta, bf16lo(cw.y)),
                                              epi_value(a[3], alpha, true, p.beta, bf16hi(cw.y)));
                            o.z = pack_bf16x2(epi_value(a[4], alpha, true, p.beta, bf16lo(cw.z)),
                                              epi_value(a[5], alpha, true, p.beta, bf16hi(cw.z)));
                            o.w = pack_bf16x2(epi_value(a[6], alpha, true, p.beta, bf16lo(cw.w)),
                                              epi_value(a[7], alpha, true, p.beta, bf16hi(cw.w)));
                        }
                        *cell = o;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (y < p.M && x < p.n_tma) tma_store_2d(&tma_d, slice, (int32_t)x, (int32_t)y);
                        bulk_commit_group();
                    }
                    store_round_tail(p, slice, lane, row, x, p.out_fp32 ? 32u : 64u);
                }
            } else if (p.tma_store && !p.out_fp32) {
                // All 128 columns are loaded under one wait and the
                // accumulator goes back to the MMAs at once; then two rounds
                // of 64 columns through this warp's 4 KiB slice of the staging
                // buffer (32 rows x 128 bytes, 128-byte swizzle).
                uint8_t* slice = staging + (half * 4 + q) * 4096u;
                uint32_t packed2[2][32];
                {
                    uint32_t v[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, v[c]);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(leader_acc_empty);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t cw[16];
                        if constexpr (has_c) {
                            // one chunk of C in flight at a time (registers)
                            asm volatile("" ::: "memory");
                            load_c_bf16x32(p, row, nbase + 32 * c, cw);
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            packed2[c >> 1][16 * (c & 1) + i] =
                                pack_bf16x2(epi_value(v[c][2 * i], alpha, has_c, p.beta, bf16lo(cw[i])),
                                            epi_value(v[c][2 * i + 1], alpha, has_c, p.beta, bf16hi(cw[i])));
                    }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t* packed = packed2[r];
                    // the slice's previous store must have read it
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<uint4*>(slice + lane * 128u + ((uint32_t)i ^ (lane & 7u)) * 16u) =
                            make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t y = row0 + q * 32, x = nbase + r * 64;
                        if (y < p.M && x < p.n_tma) tma_store_2d(&tma_d, slice, (int32_t)x, (int32_t)y);
                        bulk_commit_group();
                    }
                    store_round_tail(p, slice, lane, row, nbase + r * 64, 64u);
                    // the slice now holds this warp's 32 rows x 64 columns: read
                    // it back by columns for the output's amax
                    if constexpr (kAmax) slice_amax(slice, lane, p, amax_plain, amax_rht);
                }
            } else if (p.tma_store && p.out_fp32) {
                // FP32: all 128 columns loaded under one wait, the
                // accumulator handed back, then four rounds of 32 columns
                // through this warp's 4 KiB slice (32 rows x 128 bytes,
                // 128-byte swizzle).
                uint8_t* slice = staging + (half * 4 + q) * 4096u;
                uint32_t v[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, v[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(leader_acc_empty);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float cf[32];
                    if constexpr (has_c) load_c_f32x32(p, row, nbase + 32 * c, cf);
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<uint4*>(slice + lane * 128u + ((uint32_t)i ^ (lane & 7u)) * 16u) =
                            make_uint4(__float_as_uint(epi_value(v[c][4 * i], alpha, has_c, p.beta, cf[4 * i])),
                                       __float_as_uint(epi_value(v[c][4 * i + 1], alpha, has_c, p.beta, cf[4 * i + 1])),
                                       __float_as_uint(epi_value(v[c][4 * i + 2], alpha, has_c, p.beta, cf[4 * i + 2])),
                                       __float_as_uint(epi_value(v[c][4 * i + 3], alpha, has_c, p.beta, cf[4 * i + 3])));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t y = row0 + q * 32, x = nbase + (uint32_t)c * 32u;
                        if (y < p.M && x < p.n_tma) tma_store_2d(&tma_d, slice, (int32_t)x, (int32_t)y);
                        bulk_commit_group();
                    }
                    store_round_tail(p, slice, lane, row, nbase + (uint32_t)c * 32u, 32u);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const uint32_t n0 = nbase + 32 * c;
                    if (n0 >= p.N) break;   // warp-uniform
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, v);
                    tmem_ld_wait();
                    if (row >= p.M) continue;
                    if (p.out_fp32) {
                        float* dst = reinterpret_cast<float*>(p.d) + (int64_t)row * p.ldd + n0;
                        float cf[32];
                        if constexpr (has_c) load_c_f32x32(p, row, n0, cf);
                        if (p.vec_store && n0 + 32 <= p.N) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                store_out(reinterpret_cast<float4*>(dst + i),
                                          make_float4(epi_value(v[i], alpha, has_c, p.beta, cf[i]),
                                                      epi_value(v[i + 1], alpha, has_c, p.beta, cf[i + 1]),
                                                      epi_value(v[i + 2], alpha, has_c, p.beta, cf[i + 2]),
                                                      epi_value(v[i + 3], alpha, has_c, p.beta, cf[i + 3])),
                                          p.xd);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (n0 + i < p.N) store_out(dst + i, epi_value(v[i], alpha, has_c, p.beta, cf[i]), p.xd);
                        }
                    } else {
                        uint16_t* dst = reinterpret_cast<uint16_t*>(p.d) + (int64_t)row * p.ldd + n0;
                        uint32_t packed[16], cw[16];
                        if constexpr (has_c) load_c_bf16x32(p, row, n0, cw);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            packed[i] = pack_bf16x2(epi_value(v[2 * i], alpha, has_c, p.beta, bf16lo(cw[i])),
                                                    epi_value(v[2 * i + 1], alpha, has_c, p.beta, bf16hi(cw[i])));
                        if (p.vec_store && n0 + 32 <= p.N) {
#pragma unroll
                            for (int i = 0; i < 16; i += 4)
                                store_out(reinterpret_cast<uint4*>(dst + 2 * i),
                                          make_uint4(packed[i], packed[i + 1], packed[i + 2], packed[i + 3]), p.xd);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (n0 + i < p.N)
                                    store_out(dst + i, (uint16_t)((packed[i / 2] >> (16 * (i & 1))) & 0xFFFFu), p.xd);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(leader_acc_empty);
            }
            ++tiles_done;
        }
        if (p.tma_store && lane == 0) bulk_wait_all();
        if constexpr (kAmax) {
            amax_plain = warp_max(amax_plain);
            amax_rht = warp_max(amax_rht);
            if (lane == 0) {
                // non-negative floats order like their bit patterns
                atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(amax_plain));
                atomicMax(reinterpret_cast<unsigned int*>(p.amax_out) + 1,
                          __float_as_uint(__fmul_rn(amax_rht, 0.25f)));
            }
        }
    }

    // neither CTA frees tensor memory or exits while its peer may still use it
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host ---
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

// Scale map over the tile layout viewed as [row tile][4-scale group][128
// words]: one box is 4 groups (256 of K) of 1 or 2 row tiles.  Boxes past the
// last group or row tile read as zero.
bool make_scale_map(CUtensorMap* map, const GemmOperand& op, uint32_t box_row_tiles) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t groups = (uint64_t)((op.cols + 63) / 64), row_tiles = (uint64_t)((op.rows + 127) / 128);
    const cuuint64_t dims[3] = {128, (cuuint64_t)groups, (cuuint64_t)row_tiles};
    const cuuint64_t strides[2] = {512, (cuuint64_t)(groups * 512)};
    const cuuint32_t box[3] = {128, (cuuint32_t)kKStepsPerStage, box_row_tiles};
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(op.scales), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map: 128-byte x 32-row boxes (64 BF16 or 32 FP32 columns), 128-byte
// swizzle.
bool make_output_map(CUtensorMap* map, void* d, int64_t M, int64_t N, int64_t ldd, bool fp32) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)(ldd * (fp32 ? 4 : 2))};
    const cuuint32_t box[2] = {fp32 ? 32u : 64u, 32};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, dims, strides, box,
              elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a BF16 [rows][ld] matrix, 64 columns (128 bytes) by 128 rows
// per box with the 128-byte swizzle: the low-rank operands' K-major tiles.
bool make_bf16_rows_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// U'[m][k] = bf16(RN(U[m][k] * g)), g = RN(beta / RN(s_gA * s_gB)): the
// low-rank term rides on the accumulator that the epilogue multiplies by
// s_gA * s_gB.
__global__ void lora_prescale_kernel(const uint16_t* __restrict__ u, int64_t ldu, int64_t rows, int64_t r,
                                     float beta, const float* sga, const float* sgb, uint16_t* __restrict__ out) {
    const float g = __fdiv_rn(beta, __fmul_rn(*sga, *sgb));
    const int64_t n = rows * r;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / r, col = i - row * r;
        const float x = __uint_as_float((uint32_t)u[row * ldu + col] << 16);
        const __nv_bfloat16 h = __float2bfloat16_rn(__fmul_rn(x, g));
        out[i] = *reinterpret_cast<const uint16_t*>(&h);
    }
}

cudaError_t launch_lora_prescale(const void* u, int64_t ldu, int64_t rows, int64_t r, float beta, const float* sga,
                                 const float* sgb, void* out, cudaStream_t stream) {
    const int64_t n = rows * r;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 4 * device_sm_count()) blocks = 4 * device_sm_count();
    if (blocks < 1) blocks = 1;
    lora_prescale_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(u), ldu, rows, r, beta, sga, sgb,
                                                     static_cast<uint16_t*>(out));
    return cudaGetLastError();
}

// The kernel's warp groups trade registers with setmaxnreg against a launch
// allocation of 128 per thread (512 threads); a build that allocated fewer
// would leave the epilogue's setmaxnreg.inc waiting, so it is not launched.
bool register_split_ok() {
    static int ok = -1;
    if (ok < 0) {
        cudaFuncAttributes f0, f1;
        cudaFuncAttributes f2;
        ok = (cudaFuncGetAttributes(&f0, gemm_nvf4_kernel<kEpiPlain>) == cudaSuccess &&
              cudaFuncGetAttributes(&f1, gemm_nvf4_kernel<kEpiAmax>) == cudaSuccess &&
              cudaFuncGetAttributes(&f2, gemm_nvf4_kernel<kEpiC>) == cudaSuccess &&
              f0.numRegs * kThreads >= 128 * (64 + 72) + 256 * 184 &&
              f1.numRegs * kThreads >= 128 * (64 + 72) + 256 * 184 &&
              f2.numRegs * kThreads >= 128 * (64 + 72) + 256 * 184)
                 ? 1
                 : 0;
    }
    return ok == 1;
}

// Number of CTA pairs that can be resident at once (cached per device).
int max_active_pairs() {
    static int pairs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (pairs[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (unsigned)(device_sm_count() / 2), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_nvf4_kernel<kEpiPlain>, &cfg) != cudaSuccess || n < 1)
            n = device_sm_count() / 2;
        pairs[dev] = n > 0 ? n : 1;
    }
    return pairs[dev];
}

}  // namespace

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
                        cudaStream_t stream, const LowRank* lora, float* amax_out, uint32_t rht_mask,
                        const Axpby* axpby) {
    static bool attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_nvf4_kernel<kEpiPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_nvf4_kernel<kEpiAmax>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_nvf4_kernel<kEpiC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    if (!register_split_ok()) return cudaErrorInvalidConfiguration;
    CUtensorMap ma, mb, msa, msb, md;
    if (!make_codes_map(&ma, a, kCtaM) || !make_codes_map(&mb, b, kCtaN) || !make_scale_map(&msa, a, 1) ||
        !make_scale_map(&msb, b, 2))
        return cudaErrorInvalidValue;
    Params p{};
    p.M = (uint32_t)a.rows;
    p.N = (uint32_t)b.rows;
    p.m_tiles = (uint32_t)((a.rows + kPairM - 1) / kPairM);
    p.n_tiles = (uint32_t)((b.rows + kBN - 1) / kBN);
    p.ksteps = (uint32_t)((a.cols + 63) / 64);
    p.kstages = (p.ksteps + kKStepsPerStage - 1) / kKStepsPerStage;
    p.last_nk = p.ksteps - (p.kstages - 1) * kKStepsPerStage;
    p.n_fast = b.rows <= a.rows ? 1 : 0;   // B is the smaller operand: keep it in L2
    p.sga = a.sg;
    p.sgb = b.sg;
    p.d = d;
    p.ldd = ldd;
    p.out_fp32 = out_fp32 ? 1 : 0;
    p.xd = extent_rows(d, a.rows, ldd * (out_fp32 ? 4 : 2), b.rows * (out_fp32 ? 4 : 2));
    p.alpha = 1.0f;
    p.timeout_ns = kTimeoutNs;
    {
        // a fault armed by the test support entry point applies to this launch only
        const uint64_t armed = g_armed_fault_ns.exchange(0);
        if (armed) {
            p.timeout_ns = armed;
            p.withhold = 1;
        }
    }
    const int64_t esz = out_fp32 ? 4 : 2;
    if (axpby) {
        // the C term goes with the plain product only
        if (lora || amax_out) return cudaErrorInvalidValue;
        p.alpha = axpby->alpha;
        p.c = axpby->c;
        p.ldc = axpby->ldc;
        p.beta = axpby->beta;
        p.c_vec = ((reinterpret_cast<uintptr_t>(axpby->c) & 15u) == 0 && (axpby->ldc * esz) % 16 == 0) ? 1 : 0;
    }
    p.vec_store = ((reinterpret_cast<uintptr_t>(d) & 15u) == 0 && (ldd * esz) % 16 == 0) ? 1 : 0;
    // the D map stops at the last whole 16-byte piece of a row (a TMA store
    // writes whole pieces); the columns after it go out by the lanes' stores
    p.n_tma = (uint32_t)(out_fp32 ? (b.rows & ~int64_t(3)) : (b.rows & ~int64_t(7)));
    p.tma_store = (p.vec_store && make_output_map(&md, d, a.rows, p.n_tma > 0 ? p.n_tma : b.rows, ldd, out_fp32))
                      ? 1
                      : 0;
    if (!p.tma_store) md = ma;   // unused by the kernel; any valid map
    if (amax_out) {
        // the amax is taken in the BF16 TMA-store epilogue
        if (out_fp32 || !p.tma_store) return cudaErrorInvalidValue;
        const cudaError_t e = cudaMemsetAsync(amax_out, 0, 2 * sizeof(float), stream);
        if (e != cudaSuccess) return e;
        p.amax_out = amax_out;
        for (int i = 0; i < 16; ++i) p.rht_sgn[i] = ((rht_mask >> i) & 1u) ? 0x80008000u : 0u;
    }
    CUtensorMap mu = ma, mv = ma;  // low-rank operands (unused by the kernel otherwise; any valid map)
    p.c_staged = (p.c && p.c_vec && p.tma_store) ? 1 : 0;
    if (lora) {
        if (!make_bf16_rows_map(&mu, lora->u_scaled, a.rows, lora->r, lora->r) ||
            !make_bf16_rows_map(&mv, lora->v, b.rows, lora->r, lora->ldv))
            return cudaErrorInvalidValue;
        p.lora_stages = (uint32_t)(lora->r / 64);
        // U' = U * (beta / (s_gA s_gB)), so that the epilogue's factor
        // s_gA s_gB leaves beta * U V^T
        const cudaError_t e = launch_lora_prescale(lora->u, lora->ldu, a.rows, lora->r, lora->beta, a.sg, b.sg,
                                                   lora->u_scaled, stream);
        if (e != cudaSuccess) return e;
    }
    const uint32_t tiles = p.m_tiles * p.n_tiles;
    const uint32_t pairs = (uint32_t)max_active_pairs();
    const int grid = 2 * (int)(tiles < pairs ? tiles : pairs);
    if (p.amax_out)
        gemm_nvf4_kernel<kEpiAmax><<<grid, kThreads, kSmemBytes, stream>>>(ma, mb, msa, msb, md, mu, mv, p);
    else if (p.c)
        gemm_nvf4_kernel<kEpiC><<<grid, kThreads, kSmemBytes, stream>>>(ma, mb, msa, msb, md, mu, mv, p);
    else
        gemm_nvf4_kernel<kEpiPlain><<<grid, kThreads, kSmemBytes, stream>>>(ma, mb, msa, msb, md, mu, mv, p);
    return cudaGetLastError();
}

void arm_gemm_fault(uint64_t timeout_ns) { g_armed_fault_ns.store(timeout_ns); }

cudaError_t gemm_read_and_clear_status(unsigned int* status) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) e = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof zero);
    *status = v;
    return e;
}

cudaError_t gemm_bounds_read_and_clear(uint64_t* n) { return bounds_read_and_clear_local(n); }

}  // namespace nvfp4
