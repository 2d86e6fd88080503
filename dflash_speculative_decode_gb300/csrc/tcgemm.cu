// tcgemm.cu -- the Q4_1 product at many rows (M >= 128: prompt ingest) on the tcgen05 tensor cores.
//
// At a few rows the product streams its weights once and is bound by HBM (gemm.cu). Once a pass carries
// hundreds of rows the same product is a dense contraction, and it runs here: the weights are expanded
// to bf16 once per call, and a tcgen05 kernel multiplies them with the rows, accumulating in tensor
// memory (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass", "What changes"
// item 1: the prompt goes through the same layer products as a verify, in chunks of rows).
//
// Precision. A Q4_1 weight w = d q + m (fp16 d and m, q in 0..15) is formed in fp32 (exact: d q has at
// most 15 significant bits) and split into bf16 hi + lo with w - (hi + lo) within 2^-17 |w|; the fp32
// rows are split the same way. The product adds hi*hi + hi*lo + lo*hi (the lo*lo term lies below fp32
// rounding) in fp32 in tensor memory, so a result carries about the error of an fp32 dot product.
//
// Kernel (k_tc_gemm). A tile is 128 output columns x 128 rows; one persistent CTA per SM takes every
// G-th tile. Per stage of 64 inputs the TMA loads four 16 KB tiles (weight hi, weight lo, row hi, row
// lo), each 128 rows x 128 bytes in the 128-byte swizzle the MMA's shared-memory descriptors name; three
// stages are in flight, across tile boundaries. Warp 0 issues the copies, warp 1 owns the tensor memory
// and one of its lanes issues the MMAs (M = 128, N = 128, K = 16; twelve per stage) into one of two
// accumulators, warps 2-5 read the other one (tcgen05.ld, one 32-lane quarter each) and store the fp32
// result. Every wait on an mbarrier is bounded; a wait that gives up stops the CTA's issuing, drains
// what is in flight, frees the tensor memory and sets the error word.
#include <cuda.h>   // CUtensorMap and its enums (types only: the encoder is looked up at run time)

#include "common.cuh"
#include "dfl.h"

namespace dfl {

constexpr int kTcM = 128;                            // output columns per CTA (the MMA's M)
constexpr int kTcN = 128;                            // rows per CTA (the MMA's N)
constexpr int kTcK = 64;                             // inputs per stage: one 128-byte swizzle row of bf16
constexpr int kTcStages = 3;
constexpr int kTcTile = 128 * kTcK * 2;              // bytes of one operand tile (16 KB)
constexpr int kTcStageBytes = 4 * kTcTile;           // weight hi, weight lo, rows hi, rows lo
constexpr int kTcThreads = 192;                      // warp 0 copies, warp 1 MMAs, warps 2-5 epilogue
constexpr int kTcSmem = kTcStages * kTcStageBytes + 1024;   // + slack to align the ring to 1024 bytes
constexpr int kTcTmemCols = 2 * kTcN;                // two fp32 accumulators of 128 lanes x 128 columns

// ---------------------------------------------------------------------------------------------------
// operand preparation
// ---------------------------------------------------------------------------------------------------
__device__ __forceinline__ void split_bf16(float x, uint16_t &hi, uint16_t &lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    hi = *reinterpret_cast<const uint16_t *>(&h);
    lo = *reinterpret_cast<const uint16_t *>(&l);
}

// Weights: the tile image (16 columns x 64 inputs per 640-byte tile, codes in the lane order of
// gemm.cu) -> wh, wl bf16 [N][Kp] (row n = output column n, Kp = K padded to 64; the padding is 0).
// One warp per tile: each lane expands its 16 bytes of codes (two adjacent inputs of 16 column pairs)
// into shared memory, then the warp writes the tile's 16 rows of 128 bytes (hi and lo) with 16-byte
// stores, eight lanes per row.
constexpr int kDqWarps = 8;
constexpr int kDqPitch = 72;   // bf16 per staged row: 144 bytes, so the lanes' 4-byte writes hit 32 banks
__global__ void __launch_bounds__(kDqWarps * 32) k_tc_dequant(const uint8_t *__restrict__ img, int N, int C,
                                                              uint16_t *__restrict__ wh, uint16_t *__restrict__ wl) {
    __shared__ __align__(16) uint16_t stage[kDqWarps][2][16 * kDqPitch];
    const int warp = threadIdx.x >> 5, L = threadIdx.x & 31;
    const long tile = (long)blockIdx.x * kDqWarps + warp;
    const long ntiles = (long)(N / 16) * C;
    if (tile >= ntiles) return;   // whole warps leave together
    const int nt = int(tile / C), c = int(tile % C);
    const int g = L >> 2, t = L & 3;
    const uint8_t *src = img + tile * 640;
    const uint4 words = *reinterpret_cast<const uint4 *>(src + 16 * L);
    const uint4 dm = *reinterpret_cast<const uint4 *>(src + 512 + 16 * g);   // (n0,b0) (n1,b0) (n0,b1) (n1,b1)
    const uint32_t wv[4] = {words.x, words.y, words.z, words.w};
    const uint32_t dmv[4] = {dm.x, dm.y, dm.z, dm.w};
    uint16_t *sh = stage[warp][0], *sl = stage[warp][1];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint32_t w = wv[s];
        const int blk = s >> 1;   // 32-input block of the chunk
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // nibble pairs (e, e + 4) hold inputs (k, k + 1) of one column: e = 0: (g, 2t), 1: (g+8, 2t),
            // 2: (g, 2t+8), 3: (g+8, 2t+8)
            const int r = g + ((e & 1) ? 8 : 0);
            const int k = 16 * s + 2 * t + ((e & 2) ? 8 : 0);
            const uint32_t pair = dmv[2 * blk + (e & 1)];
            const float d = __half2float(__ushort_as_half(uint16_t(pair & 0xFFFFu)));
            const float m = __half2float(__ushort_as_half(uint16_t(pair >> 16)));
            const float q0 = float((w >> (4 * e)) & 15u), q1 = float((w >> (4 * e + 16)) & 15u);
            uint16_t h0, l0, h1, l1;
            split_bf16(fmaf(d, q0, m), h0, l0);
            split_bf16(fmaf(d, q1, m), h1, l1);
            *reinterpret_cast<uint32_t *>(sh + r * kDqPitch + k) = uint32_t(h0) | (uint32_t(h1) << 16);
            *reinterpret_cast<uint32_t *>(sl + r * kDqPitch + k) = uint32_t(l0) | (uint32_t(l1) << 16);
        }
    }
    __syncwarp();
    const long Kp = (long)C * 64;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int idx = it * 32 + L;              // 0..255: (array, row, 16-byte chunk)
        const int arr = idx >> 7, r = (idx >> 3) & 15, ch = idx & 7;
        const uint16_t *from = stage[warp][arr] + r * kDqPitch + 8 * ch;
        uint16_t *to = (arr ? wl : wh) + (long)(16 * nt + r) * Kp + 64 * c + 8 * ch;
        *reinterpret_cast<uint4 *>(to) = *reinterpret_cast<const uint4 *>(from);
    }
}

// Rows: fp32 x [M][K] -> xh, xl bf16 [M][Kp] (zero past K). Two inputs per thread.
__global__ void k_tc_split(const float *__restrict__ x, int M, int K, int Kp, uint16_t *__restrict__ xh,
                           uint16_t *__restrict__ xl) {
    const long i = blockIdx.x * (long)blockDim.x + threadIdx.x;   // pair index
    const long pairs = (long)M * Kp / 2;
    if (i >= pairs) return;
    const long m = (2 * i) / Kp;
    const int k = int((2 * i) % Kp);
    const float x0 = k < K ? x[m * K + k] : 0.f;
    const float x1 = k + 1 < K ? x[m * K + k + 1] : 0.f;
    uint16_t h0, l0, h1, l1;
    split_bf16(x0, h0, l0);
    split_bf16(x1, h1, l1);
    reinterpret_cast<uint32_t *>(xh)[i] = uint32_t(h0) | (uint32_t(h1) << 16);
    reinterpret_cast<uint32_t *>(xl)[i] = uint32_t(l0) | (uint32_t(l1) << 16);
}

// ---------------------------------------------------------------------------------------------------
// tcgen05, TMA and mbarrier pieces (inline PTX)
// ---------------------------------------------------------------------------------------------------
// Wait for a phase bounded by time only (used to drain copies and products already issued, which
// complete on their own whatever else went wrong). Returns false if it gave up.
__device__ __forceinline__ bool mbar_drain(uint64_t *b, unsigned parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_test(b, parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// 2-D tiled TMA load of box (x = inner coordinate, y = row) into shared memory, completing on b
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *b) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(saddr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(b))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle: rows of 128 bytes, groups
// of 8 rows 1024 bytes apart (stride byte offset), descriptor version 1, layout code 2 (128B swizzle).
// The tile must start on a 1024-byte boundary; the k-step j of 16 inputs starts 32 j bytes further.
__device__ __forceinline__ uint64_t sw128_desc(const void *tile) {
    const uint64_t a = saddr(tile);
    return ((a >> 4) & 0x3FFFull) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major, N = kTcN, M = kTcM.
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kTcN >> 3) << 17) |
                              (uint32_t(kTcM >> 4) << 24);

// D (tensor memory) = A B^T (+ D when accumulate), A = 128 x 16 and B = 128 x 16 from shared memory
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}

// one arrival on b once every MMA this thread issued before has completed
__device__ __forceinline__ void tc_commit(uint64_t *b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(b))
                 : "memory");
}

// 32 consecutive accumulator columns of this thread's lane (warp quarter w % 4 of the 128 lanes)
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct TcArgs {
    int M, N, stages;   // rows, output columns, stages of 64 inputs
    int tiles_m, tiles; // 128-row tiles, tiles in all (row tiles vary fastest)
    float *y;           // [M][N] fp32
    int *err;           // sticky error bits (kErrWaitTimeout), nullable
};

// Persistent: CTA c takes tiles c, c + G, c + 2G, ... Consecutive tiles share their weight tile (row
// tiles vary fastest), so the CTAs working at once read few weight tiles from HBM and the rows stay in
// L2. Two accumulators in tensor memory: the epilogue drains one while the products fill the other.
__global__ void __launch_bounds__(kTcThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap tw_hi, const __grid_constant__ CUtensorMap tw_lo,
              const __grid_constant__ CUtensorMap tx_hi, const __grid_constant__ CUtensorMap tx_lo, TcArgs a) {
    extern __shared__ uint8_t tc_smem_raw[];
    __shared__ __align__(8) uint64_t full[kTcStages], empty[kTcStages], accf[2], acce[2], done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued, s_consumed;
    __shared__ volatile int s_bad;
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nst = a.stages;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&full[i], 1);    // the producer's arrival (with the stage's bytes)
            mbar_init(&empty[i], 1);   // the MMA thread's commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);    // the MMA thread's commit after a tile's last stage
            mbar_init(&acce[b], 4);    // one arrival per epilogue warp once it has read the accumulator
        }
        mbar_init(&done, 1);           // the MMA thread's last commit
        s_bad = 0;
        s_issued = s_consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {   // the whole warp allocates both accumulators' columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&s_tmem)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ---- copies: every stage of every tile of this CTA, through the ring ----
        if (lane == 0) {
            int k = 0;
            bool stop = false;
            for (int t = blockIdx.x; t < a.tiles && !stop; t += gridDim.x) {
                const int m0 = (t % a.tiles_m) * kTcN, n0 = (t / a.tiles_m) * kTcM;
                for (int st = 0; st < nst; ++st, ++k) {
                    const int s = k % kTcStages;
                    if (k >= kTcStages && !mbar_wait(&empty[s], unsigned(k / kTcStages - 1) & 1u, &s_bad)) {
                        stop = true;
                        break;
                    }
                    if (s_bad) {
                        stop = true;
                        break;
                    }
                    uint8_t *sp = ring + s * kTcStageBytes;
                    mbar_expect(&full[s], unsigned(kTcStageBytes));
                    tma_load_2d(sp, &tw_hi, st * kTcK, n0, &full[s]);
                    tma_load_2d(sp + kTcTile, &tw_lo, st * kTcK, n0, &full[s]);
                    tma_load_2d(sp + 2 * kTcTile, &tx_hi, st * kTcK, m0, &full[s]);
                    tma_load_2d(sp + 3 * kTcTile, &tx_lo, st * kTcK, m0, &full[s]);
                }
            }
            s_issued = k;
        }
    } else if (warp == 1) {
        // ---- products: tile li into accumulator li % 2 ----
        if (lane == 0) {
            int k = 0, li = 0;
            bool stop = false;
            for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++li) {
                const int b = li & 1;
                const uint32_t d = tmem + uint32_t(b * kTcN);
                if (li >= 2 && !mbar_wait(&acce[b], unsigned(li / 2 - 1) & 1u, &s_bad)) break;
                tc_fence_after();
                for (int st = 0; st < nst; ++st, ++k) {
                    const int s = k % kTcStages;
                    if (!mbar_wait(&full[s], unsigned(k / kTcStages) & 1u, &s_bad)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *sp = ring + s * kTcStageBytes;
                    const uint64_t dwh = sw128_desc(sp), dwl = sw128_desc(sp + kTcTile);
                    const uint64_t dxh = sw128_desc(sp + 2 * kTcTile), dxl = sw128_desc(sp + 3 * kTcTile);
#pragma unroll
                    for (int j = 0; j < kTcK / 16; ++j) {
                        const uint64_t o = uint64_t(2 * j);   // 32 bytes further, in 16-byte units
                        tc_mma(d, dwh + o, dxh + o, (st > 0 || j > 0) ? 1u : 0u);
                        tc_mma(d, dwh + o, dxl + o, 1u);
                        tc_mma(d, dwl + o, dxh + o, 1u);
                    }
                    tc_commit(&empty[s]);   // the stage may be refilled once these products are done
                }
                if (stop) break;
                tc_commit(&accf[b]);        // the tile's accumulator is complete
            }
            s_consumed = k;
            tc_commit(&done);               // every product issued (also on the error path)
        }
        __syncwarp();
    } else {
        // ---- epilogue: warps 2..5, lane quarter warp % 4 ----
        const int q = warp & 3;
        int li = 0;
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++li) {
            const int b = li & 1;
            const bool ok = mbar_wait(&accf[b], unsigned(li / 2) & 1u, &s_bad);
            tc_fence_after();
            // tcgen05.ld is warp-collective: the whole warp reads, or none of it
            if (!__all_sync(0xffffffffu, ok && !s_bad)) break;
            const int m0 = (t % a.tiles_m) * kTcN, n0 = (t / a.tiles_m) * kTcM;
            const int f = n0 + 32 * q + lane;
#pragma unroll 1
            for (int c0 = 0; c0 < kTcN; c0 += 32) {
                uint32_t r[32];
                tc_ld32(tmem + uint32_t(b * kTcN) + (uint32_t(32 * q) << 16) + uint32_t(c0), r);
                if (f < a.N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int m = m0 + c0 + j;
                        if (m < a.M) a.y[(long)m * a.N + f] = __uint_as_float(r[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);   // accumulator b may be overwritten
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // every commit lands before the memory is released; after a wait gave up, also every copy
        // already issued
        if (s_bad)
            for (int k = s_consumed; k < s_issued; ++k) mbar_drain(&full[k % kTcStages], unsigned(k / kTcStages) & 1u);
        if (!mbar_drain(&done, 0u)) s_bad = 1;
        if (s_bad && a.err) atomicOr(a.err, kErrWaitTimeout);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// bf16 matrix [rows][Kp] (Kp a multiple of 64, base 16-byte aligned) as 64 x 128 boxes in the 128-byte
// swizzle; rows past the end read as zero
static bool bf16_map(CUtensorMap *map, const void *base, long rows, int Kp) {
    const EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(Kp), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(Kp) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kTcK), 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// scratch: [256-byte header: error word][wh][wl][xh][xl], each region 1024-byte aligned
struct TcScratch {
    size_t wbytes, xbytes, total;
};
static TcScratch tc_scratch(int K, int N, int M) {
    const size_t Kp = (size_t)padded_k(K);
    TcScratch s;
    s.wbytes = (N * Kp * 2 + 1023) / 1024 * 1024;
    s.xbytes = ((size_t)M * Kp * 2 + 1023) / 1024 * 1024;
    s.total = 1024 + 2 * s.wbytes + 2 * s.xbytes;
    return s;
}

static bool tc_shape_ok(int K, int N, int M) {
    return K >= 32 && K % 32 == 0 && N >= 32 && N % 32 == 0 && M >= 1 && M <= (1 << 20) && (long)K * N < (1L << 31);
}

size_t tc_gemm_scratch_bytes(int K, int N, int M) { return tc_shape_ok(K, N, M) ? tc_scratch(K, N, M).total : 0; }

// Expand the weights, split the rows and run the product (three launches on s). The scratch's first
// 1024 bytes are not used here (the entry point keeps its error word there).
cudaError_t launch_tc_gemm(const uint8_t *img, int K, int N, const float *x, int M, float *y, void *scratch,
                           int *err, cudaStream_t s) {
    if (!tc_shape_ok(K, N, M) || !img || !x || !y || !scratch || (reinterpret_cast<uintptr_t>(scratch) & 1023))
        return cudaErrorInvalidValue;
    const TcScratch ts = tc_scratch(K, N, M);
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    const int Kp = padded_k(K), C = Kp / 64;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    uint16_t *wh = reinterpret_cast<uint16_t *>(base + 1024);
    uint16_t *wl = reinterpret_cast<uint16_t *>(base + 1024 + ts.wbytes);
    uint16_t *xh = reinterpret_cast<uint16_t *>(base + 1024 + 2 * ts.wbytes);
    uint16_t *xl = reinterpret_cast<uint16_t *>(base + 1024 + 2 * ts.wbytes + ts.xbytes);
    CUtensorMap mwh, mwl, mxh, mxl;
    if (!bf16_map(&mwh, wh, N, Kp) || !bf16_map(&mwl, wl, N, Kp) || !bf16_map(&mxh, xh, M, Kp) ||
        !bf16_map(&mxl, xl, M, Kp))
        return cudaErrorInvalidValue;
    static bool attr[kMaxDevices] = {};
    if (!attr[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(k_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    const long wtiles = (long)(N / 16) * C;
    k_tc_dequant<<<unsigned((wtiles + kDqWarps - 1) / kDqWarps), kDqWarps * 32, 0, s>>>(img, N, C, wh, wl);
    const long xpairs = (long)M * Kp / 2;
    k_tc_split<<<unsigned((xpairs + 255) / 256), 256, 0, s>>>(x, M, K, Kp, xh, xl);
    static int sms[kMaxDevices] = {};
    if (!sms[dev] && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    TcArgs a;
    a.M = M;
    a.N = N;
    a.stages = C;
    a.tiles_m = (M + kTcN - 1) / kTcN;
    a.tiles = a.tiles_m * ((N + kTcM - 1) / kTcM);
    a.y = y;
    a.err = err;
    const int grid = a.tiles < sms[dev] ? a.tiles : sms[dev];   // persistent: one CTA per SM
    k_tc_gemm<<<grid, kTcThreads, kTcSmem, s>>>(mwh, mwl, mxh, mxl, a);
    return cudaGetLastError();
}

}  // namespace dfl

using namespace dfl;

extern "C" {

int64_t dfl_q41_gemm_tc_scratch_bytes(int K, int N, int M) {
    if (!tc_shape_ok(K, N, M)) return -1;
    return (int64_t)tc_scratch(K, N, M).total;
}

int dfl_q41_gemm_tc(const void *img, int K, int N, const float *x, int M, float *y, void *scratch,
                    size_t scratch_bytes, void *stream) {
    if (!tc_shape_ok(K, N, M) || !img || !x || !y || !scratch) return DFL_E_INVALID_ARG;
    if (scratch_bytes < tc_scratch(K, N, M).total || (reinterpret_cast<uintptr_t>(scratch) & 1023))
        return DFL_E_INVALID_ARG;
    const cudaError_t e = launch_tc_gemm(static_cast<const uint8_t *>(img), K, N, x, M, y, scratch,
                                         static_cast<int *>(scratch), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DFL_OK : DFL_E_CUDA;
}

}  // extern "C"
