// gemm.cu -- the skinny products of the step (M = 1..16 rows).
//
// Every projection of the batched verify and of the draft is one M-row product over a weight image
// streamed once from HBM (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass",
// "What changes": a verify of k rows used to cost k passes over the weights). Weights are Q4_1
// (model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", spec table: "5 bits per weight with scales and
// minimums") except fc and the head, which are bf16.
//
// Weight layout. A matrix of K inputs x N outputs is cut into tiles of 16 output columns x 64 inputs;
// tile (nt, c) of a matrix with C = ceil(K/64) chunks sits at (nt*C + c) * tile_bytes. Inside a tile
// the data is ordered by the lane that consumes it as the A operand of mma.m16n8k16 (rows = output
// columns, columns = inputs):
//   Q4_1 (640 B): lane L = 4g + t holds 16 B of codes at 16L: word s (k-step s, inputs 16s..16s+15)
//     packs, low to high nibble, q(g,2t) q(g+8,2t) q(g,2t+8) q(g+8,2t+8) q(g,2t+1) q(g+8,2t+1)
//     q(g,2t+9) q(g+8,2t+9), so shifting by 0/4/8/12 and masking 0x000F000F gives the four A registers.
//     Bytes 512..639: for g = 0..7, 16 B of (d, m) fp16 pairs for columns g, g+8 of the tile's two
//     32-input blocks.
//   bf16 (2048 B): k-step s at 512*s, lane L's 16 B = its four A registers.
// Activations arrive in the operand format of common.cuh (bf16 hi + lo fragments in lane order and
// per-16 sums), so a warp loads its B fragment of a k-step with one 16-byte load.
//
// Q4_1 product per 32-block b: y += d_b * sum_k x_k q_k + m_b * sum_k x_k, with q entering the tensor
// core exactly (integers 0..15 are exact in bf16) and the per-block scale applied in fp32.
//
// Work split (stream-K). Units = (quad of four 32-column groups, 64-input chunk). A persistent grid
// of one wave takes equal contiguous unit ranges; the four warps of a CTA take the four column groups
// of a quad, so they read the same activation chunks. A column group whose chunks span several CTAs
// gets one partial sum per CTA ("segment"); the last segment to finish (arrival counter) adds them in
// segment order and applies the epilogue. Segments depend on K, N and the grid only, so a row's
// result never depends on how many rows the pass carries.
#include <algorithm>

#include "common.cuh"
#include "rowstep.cuh"

namespace dfl {

// compute warps of a product CTA: four column groups x kGemmPar chunk parities
constexpr int kGemmWarps = 8, kGemmThreads = kGemmWarps * 32, kGemmPar = kGemmWarps / 4;


// ---------------------------------------------------------------------------------------------------
// packing
// ---------------------------------------------------------------------------------------------------
__global__ void k_pack_q41(const uint8_t *__restrict__ src, int K, int N, int C, uint8_t *__restrict__ img) {
    const long tid = blockIdx.x * (long)blockDim.x + threadIdx.x;
    const long ntiles = (long)(N / 16) * C;
    if (tid >= ntiles * 32) return;
    const int L = int(tid & 31);
    const long tile = tid >> 5;
    const int nt = int(tile / C), c = int(tile % C);
    const int g = L >> 2, t = L & 3;
    const int nb = K / 32;
    const int n0 = 16 * nt + g, n1 = n0 + 8;
    auto code = [&](int n, int k) -> uint32_t {
        if (k >= K) return 0u;
        const uint8_t *blk = src + ((long)n * nb + k / 32) * 20;
        const int i = k & 31;
        const uint8_t by = blk[4 + i / 2];
        return (i & 1) ? uint32_t(by >> 4) : uint32_t(by & 15);
    };
    uint32_t w[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int kb = 64 * c + 16 * s;
        w[s] = code(n0, kb + 2 * t) | (code(n1, kb + 2 * t) << 4) | (code(n0, kb + 2 * t + 8) << 8) |
               (code(n1, kb + 2 * t + 8) << 12) | (code(n0, kb + 2 * t + 1) << 16) |
               (code(n1, kb + 2 * t + 1) << 20) | (code(n0, kb + 2 * t + 9) << 24) |
               (code(n1, kb + 2 * t + 9) << 28);
    }
    uint8_t *dst = img + tile * 640;
    *reinterpret_cast<uint4 *>(dst + 16 * L) = make_uint4(w[0], w[1], w[2], w[3]);
    if (t == 0) {
        auto dm = [&](int n, int b) -> uint32_t {
            if (b >= nb) return 0u;
            return *reinterpret_cast<const uint32_t *>(src + ((long)n * nb + b) * 20);
        };
        *reinterpret_cast<uint4 *>(dst + 512 + 16 * g) =
            make_uint4(dm(n0, 2 * c), dm(n1, 2 * c), dm(n0, 2 * c + 1), dm(n1, 2 * c + 1));
    }
}

__global__ void k_pack_bf16(const uint16_t *__restrict__ src, int K, int N, int C, uint8_t *__restrict__ img) {
    const long tid = blockIdx.x * (long)blockDim.x + threadIdx.x;
    const long ntiles = (long)(N / 16) * C;
    if (tid >= ntiles * 128) return;
    const int L = int(tid & 31);
    const int s = int((tid >> 5) & 3);
    const long tile = tid >> 7;
    const int nt = int(tile / C), c = int(tile % C);
    const int g = L >> 2, t = L & 3;
    const int n0 = 16 * nt + g, n1 = n0 + 8;
    const int kb = 64 * c + 16 * s;
    auto pair = [&](int n, int k) -> uint32_t {
        if (k >= K) return 0u;
        const uint16_t *p = src + (long)n * K + k;
        return uint32_t(p[0]) | (uint32_t(p[1]) << 16);
    };
    uint4 v = make_uint4(pair(n0, kb + 2 * t), pair(n1, kb + 2 * t), pair(n0, kb + 2 * t + 8), pair(n1, kb + 2 * t + 8));
    *reinterpret_cast<uint4 *>(img + tile * 2048 + 512 * s + 16 * L) = v;
}

cudaError_t launch_pack_q41(const uint8_t *src, int K, int N, uint8_t *img, cudaStream_t s) {
    const int C = padded_k(K) / 64;
    const long threads = (long)(N / 16) * C * 32;
    k_pack_q41<<<unsigned((threads + 255) / 256), 256, 0, s>>>(src, K, N, C, img);
    return cudaGetLastError();
}

cudaError_t launch_pack_bf16(const uint16_t *src, int K, int N, uint8_t *img, cudaStream_t s) {
    const int C = padded_k(K) / 64;
    const long threads = (long)(N / 16) * C * 128;
    k_pack_bf16<<<unsigned((threads + 255) / 256), 256, 0, s>>>(src, K, N, C, img);
    return cudaGetLastError();
}

// fp32 rows -> operand format (the standalone product's input)
__global__ void k_act_pack(const float *x, int M, int K, uint32_t *f, float *sums) {
    pdl_trigger();
    pdl_wait();
    const int m = blockIdx.y;
    const int k = blockIdx.x * blockDim.x + threadIdx.x;   // blockDim 256: a 16-group is one half warp
    const bool in = k < K && m < M;
    const float v = in ? x[(long)m * K + k] : 0.f;
    const float s = half_warp_sum(in ? act_store(f, K, m, k, v) : 0.f);
    if (in && (k & 15) == 0) sums[(k / 16) * kMaxRows + m] = s;
}

cudaError_t launch_act_pack(const float *x, int M, int K, uint32_t *f, float *sums, cudaStream_t s) {
    return launch_pdl(k_act_pack, dim3((K + 255) / 256, M), dim3(256), 0, s, x, M, K, f, sums);
}

// ---------------------------------------------------------------------------------------------------
// shared-memory ring
// A round is CPR consecutive chunks of one quad (CPR units; 8 for Q4_1, 4 for bf16). Its weights
// (8*CPR tiles) and activations (R = 8*MT rows x CPR chunks, plus the chunks' per-16 sums) are brought
// into one ring slot by bulk asynchronous copies, one per contiguous run, completing on the slot's
// "full" mbarrier:
//   tiles: tile (unit u, group gq, tile j) at ((2*gq + j)*CPR + u) * TB  (a group's chunks are one run)
//   rows:  row block rb (8 rows) at WB + rb * CP * 2048, chunk u at + 2048*u, k-step ks at + 512*ks,
//          row tok % 8 at + 64*(tok % 8) (the operand format's own order: one copy per row block)
//   sums:  at WB + MT * CP * 2048, 256 bytes per chunk ([4 groups][16 rows] fp32)
// ---------------------------------------------------------------------------------------------------
template <int FMT>
__host__ __device__ constexpr int cpr() { return FMT == W_Q41 ? 8 : 4; }
template <int FMT>
__host__ __device__ constexpr int xblock_bytes() { return cpr<FMT>() * 2048; }   // one row block of a round
template <int MT>
__host__ __device__ constexpr int red_bytes() { return kGemmPar * 4 * MT * 8 * 32 * 4; }   // [parity][4 groups][R][32]
template <int FMT>
__host__ __device__ constexpr int tile_bytes() { return FMT == W_Q41 ? 640 : 2048; }
template <int FMT, int MT>
__host__ __device__ constexpr int slot_bytes() {
    return (8 * cpr<FMT>() * tile_bytes<FMT>() + MT * xblock_bytes<FMT>() + cpr<FMT>() * 256 + 127) / 128 * 128;
}
constexpr int kGemmSmemBudget = 224 * 1024;
template <int FMT, int MT>
__host__ __device__ constexpr int ring_slots() {
    return (kGemmSmemBudget - red_bytes<MT>()) / slot_bytes<FMT, MT>() < 6 ? (kGemmSmemBudget - red_bytes<MT>()) / slot_bytes<FMT, MT>() : 6;
}

// two fp32 lanes at once: d = a * b + c (each lane rounded as fmaf)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

// mma.m16n8k16 bf16 with a zero accumulator
__device__ __forceinline__ void mma_bf16_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                           uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// ---------------------------------------------------------------------------------------------------
// a warp's units of one round: NU chunks (u = par + kGemmPar*i) of its column group, two 16-column tiles each
// ---------------------------------------------------------------------------------------------------
// Q4_1: the codes enter the tensor cores as 128 + q (exact in bf16), so per 32-block b
//   sum_k x_k w_k = d_b sum_k x_k (128 + q_k) + (m_b - 128 d_b) sum_k x_k,
// with sum_k x_k the per-16 sums of the operand (hi + lo) values. The NU units are independent until
// the fold, so their loads and products overlap. nblk[i]: 32-blocks of unit i inside K (0: no unit).
template <int FMT, int MT, int NU>
__device__ __forceinline__ void q41_units(float (&acc)[2][MT][4], const uint8_t *slot, int w_off, int x_off, int s_off,
                                          const int (&nblk)[NU], int lane) {
    constexpr int TB = tile_bytes<FMT>(), CP = cpr<FMT>(), XB = xblock_bytes<FMT>();
    const int t = lane & 3, g = lane >> 2;
    uint4 nb[NU][2], sc[NU][2];
#pragma unroll
    for (int i = 0; i < NU; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint8_t *w = slot + w_off + (j * CP + kGemmPar * i) * TB;
            nb[i][j] = *reinterpret_cast<const uint4 *>(w + 16 * lane);
            sc[i][j] = *reinterpret_cast<const uint4 *>(w + 512 + 16 * g);
        }
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        float c[NU][2][MT][4];
        float2 S[NU][MT];
#pragma unroll
        for (int i = 0; i < NU; ++i) {
            const float *xsum = reinterpret_cast<const float *>(slot + s_off + 256 * kGemmPar * i);
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
                const float2 s0 = *reinterpret_cast<const float2 *>(xsum + (2 * blk) * kMaxRows + 8 * tt + 2 * t);
                const float2 s1 = *reinterpret_cast<const float2 *>(xsum + (2 * blk + 1) * kMaxRows + 8 * tt + 2 * t);
                S[i][tt] = make_float2(s0.x + s1.x, s0.y + s1.y);
            }
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int ks = 2 * blk + kk;
            uint4 b[NU][MT];
            uint32_t A[NU][2][4];
#pragma unroll
            for (int i = 0; i < NU; ++i) {
#pragma unroll
                for (int tt = 0; tt < MT; ++tt)
                    b[i][tt] = *reinterpret_cast<const uint4 *>(slot + x_off + 2048 * kGemmPar * i + tt * XB + 512 * ks);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t w = ks == 0 ? nb[i][j].x : ks == 1 ? nb[i][j].y : ks == 2 ? nb[i][j].z : nb[i][j].w;
                    A[i][j][0] = nib_pair_bf16(w), A[i][j][1] = nib_pair_bf16(w >> 4);
                    A[i][j][2] = nib_pair_bf16(w >> 8), A[i][j][3] = nib_pair_bf16(w >> 12);
                }
            }
            // the hi products of every (unit, tile) first, then the lo products: consecutive products
            // feed different accumulators
#pragma unroll
            for (int i = 0; i < NU; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt) {
                        if (kk == 0) mma_bf16_z(c[i][j][tt], A[i][j][0], A[i][j][1], A[i][j][2], A[i][j][3], b[i][tt].x, b[i][tt].y);
                        else mma_bf16(c[i][j][tt], A[i][j][0], A[i][j][1], A[i][j][2], A[i][j][3], b[i][tt].x, b[i][tt].y);
                    }
#pragma unroll
            for (int i = 0; i < NU; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
                        mma_bf16(c[i][j][tt], A[i][j][0], A[i][j][1], A[i][j][2], A[i][j][3], b[i][tt].z, b[i][tt].w);
        }
#pragma unroll
        for (int i = 0; i < NU; ++i) {
            if (blk >= nblk[i]) continue;   // past K, or no unit: its registers hold nothing of use
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t dlo = blk ? sc[i][j].z : sc[i][j].x, dhi = blk ? sc[i][j].w : sc[i][j].y;
                const float2 flo = __half22float2(*reinterpret_cast<__half2 *>(&dlo));   // (d, m) of column g
                const float2 fhi = __half22float2(*reinterpret_cast<__half2 *>(&dhi));   // column g + 8
                const float mlo = fmaf(-128.f, flo.x, flo.y), mhi = fmaf(-128.f, fhi.x, fhi.y);
#pragma unroll
                for (int tt = 0; tt < MT; ++tt) {
                    float2 p0 = make_float2(acc[j][tt][0], acc[j][tt][1]), p1 = make_float2(acc[j][tt][2], acc[j][tt][3]);
                    p0 = ffma2(make_float2(flo.x, flo.x), make_float2(c[i][j][tt][0], c[i][j][tt][1]), p0);
                    p1 = ffma2(make_float2(fhi.x, fhi.x), make_float2(c[i][j][tt][2], c[i][j][tt][3]), p1);
                    p0 = ffma2(make_float2(mlo, mlo), S[i][tt], p0);
                    p1 = ffma2(make_float2(mhi, mhi), S[i][tt], p1);
                    acc[j][tt][0] = p0.x, acc[j][tt][1] = p0.y, acc[j][tt][2] = p1.x, acc[j][tt][3] = p1.y;
                }
            }
        }
    }
}

// bf16 (one unit per round): nks = k-steps inside K
template <int FMT, int MT>
__device__ __forceinline__ void bf16_unit(float (&acc)[2][MT][4], const uint8_t *slot, int w_off, int x_off, int nks, int lane) {
    constexpr int TB = tile_bytes<FMT>(), CP = cpr<FMT>(), XB = xblock_bytes<FMT>();
    const uint8_t *w0 = slot + w_off, *w1 = slot + w_off + CP * TB;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        if (ks >= nks) break;
        uint4 b[MT];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) b[tt] = *reinterpret_cast<const uint4 *>(slot + x_off + tt * XB + 512 * ks);
        const uint4 wa = *reinterpret_cast<const uint4 *>(w0 + 512 * ks + 16 * lane);
        const uint4 wb = *reinterpret_cast<const uint4 *>(w1 + 512 * ks + 16 * lane);
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
            mma_bf16(acc[0][tt], wa.x, wa.y, wa.z, wa.w, b[tt].x, b[tt].y);
            mma_bf16(acc[1][tt], wb.x, wb.y, wb.z, wb.w, b[tt].x, b[tt].y);
        }
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
            mma_bf16(acc[0][tt], wa.x, wa.y, wa.z, wa.w, b[tt].z, b[tt].w);
            mma_bf16(acc[1][tt], wb.x, wb.y, wb.z, wb.w, b[tt].z, b[tt].w);
        }
    }
}

// ---------------------------------------------------------------------------------------------------
// epilogue: plain fp32 rows, or the operand format of the next product (with its per-16 sums)
// ---------------------------------------------------------------------------------------------------
// sum over the 8 lanes with the same t (the 16 columns g, g+8 of a tile for one token)
__device__ __forceinline__ float tile_col_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
}

template <int MT, int EPI>
__device__ __forceinline__ void epilogue(const GemmArgs &a, float (&acc)[2][MT][4], int nt0, int nt1, int ng, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int tok = 8 * tt + 2 * t + h;
            const bool live = tok < a.M;
            if (EPI == EPI_F32) {
                if (!live) continue;
                float *y = a.y + (long)tok * a.ldy;
                y[16 * nt0 + g] = acc[0][tt][h];
                y[16 * nt0 + g + 8] = acc[0][tt][h + 2];
                y[16 * nt1 + g] = acc[1][tt][h];
                y[16 * nt1 + g + 8] = acc[1][tt][h + 2];
            } else if (EPI == EPI_GLU) {
                const float v0 = silu_f(acc[0][tt][h]) * acc[1][tt][h];
                const float v1 = silu_f(acc[0][tt][h + 2]) * acc[1][tt][h + 2];
                const int K = a.N / 2;
                float hl = 0.f;
                if (live) hl = act_store(a.yf, K, tok, 16 * ng + g, v0) + act_store(a.yf, K, tok, 16 * ng + g + 8, v1);
                const float s = tile_col_sum(hl);
                if (live && g == 0) a.ys[ng * kMaxRows + tok] = s;
            } else if (EPI == EPI_SILU_MUL) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int nt = j ? nt1 : nt0;
                    float hl = 0.f;
                    if (live) {
                        const uint16_t *e = a.ext + (long)tok * a.lde;
                        const float v0 = silu_f(acc[j][tt][h]) * bf16_to_f32(e[16 * nt + g]);
                        const float v1 = silu_f(acc[j][tt][h + 2]) * bf16_to_f32(e[16 * nt + g + 8]);
                        hl = act_store(a.yf, a.N, tok, 16 * nt + g, v0) + act_store(a.yf, a.N, tok, 16 * nt + g + 8, v1);
                    }
                    const float s = tile_col_sum(hl);
                    if (live && g == 0) a.ys[nt * kMaxRows + tok] = s;
                }
            }
        }
}

// ---------------------------------------------------------------------------------------------------
// the product kernel
// ---------------------------------------------------------------------------------------------------
// One CTA per SM: kGemmWarps compute warps and one copy warp. The CTA's unit range [u0, u1) is walked
// in rounds; compute warp w takes column group gq = w % 4 and the round's units par, par + kGemmPar, ...
// (par = w / 4). The copy warp fills the ring: a slot is refilled once every compute warp has released
// it ("empty" mbarrier), and the weights of the first ring_slots rounds are requested before the
// previous kernel has finished. At the end of a quad's range the parities are added in shared memory
// (in parity order); a quad split over several CTAs leaves one partial per CTA, added by the last CTA
// to finish it (order of the segments). Every split depends on K, N and the grid only, so a row's result
// never depends on how many rows the pass carries.
constexpr int kGemmBlock = kGemmThreads + 32;   // + the copy warp
static_assert(kGemmBlock == kProductRowThreads, "row step of the products");

// barrier of the 16 compute warps only
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kGemmThreads) : "memory"); }

template <int FMT, int MT, int EPI>
__global__ void __launch_bounds__(kGemmBlock, 1) k_gemm(GemmArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[8], empty[8];
    __shared__ int s_last, s_issued, s_ticket;
    __shared__ volatile int s_bad;   // set by the first bounded wait that gives up
    constexpr int R = MT * 8;
    constexpr int TB = tile_bytes<FMT>();
    constexpr int CP = cpr<FMT>();
    constexpr int NU = CP / kGemmPar;
    static_assert(CP % kGemmPar == 0, "units per warp");
    constexpr int XB = xblock_bytes<FMT>();
    constexpr int WB = 8 * CP * TB;
    constexpr int SB = slot_bytes<FMT, MT>();
    constexpr int S = ring_slots<FMT, MT>();
    static_assert(S >= 2 && S <= 8, "ring");
    float *red = reinterpret_cast<float *>(smem);               // [par][4 gq][R][32]
    uint8_t *ring = smem + red_bytes<MT>();                     // [S][SB]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int ngroups = a.N / 32;
    const int Q = (ngroups + 3) / 4;
    const long U = (long)Q * a.C;
    const int G = gridDim.x;
    const int K16 = a.K / 16;
    const long u0 = (long)blockIdx.x * U / G, u1 = (long)(blockIdx.x + 1) * U / G;

    // a round: chunks c .. min(c + CP, ce) - 1 of quad q
    struct Rd {
        int q, c, ce;
    };
    auto rd_at_quad = [&](Rd &r, int q, int c) {
        r.q = q;
        r.c = c;
        const long e = u1 - (long)q * a.C;
        r.ce = int(e < a.C ? e : a.C);
    };
    auto rd_valid = [&](const Rd &r) { return (long)r.q * a.C + r.c < u1; };
    auto rd_next = [&](Rd &r) {
        if (r.c + CP < r.ce) r.c += CP;
        else rd_at_quad(r, r.q + 1, 0);
    };
    auto tile_of = [&](int ng, int j) { return EPI == EPI_GLU ? (j ? ng + ngroups : ng) : 2 * ng + j; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 2);            // weights arrival + activations arrival (+ their bytes)
            mbar_init(&empty[i], kGemmWarps);  // one arrival per compute warp
        }
        s_bad = 0;
        s_last = 0;
        s_issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    if (warp == kGemmWarps) {
        // ---- copy warp ----
        auto issue_w = [&](const Rd &r, int sl) {   // the weights of round r into slot sl
            const int nc = r.ce - r.c < CP ? r.ce - r.c : CP;
            const int live = ngroups - 4 * r.q < 4 ? ngroups - 4 * r.q : 4;
            if (lane == 0) mbar_expect(&full[sl], unsigned(2 * live * nc * TB));
            __syncwarp();
            if (lane < 2 * live) {
                const int gg = lane >> 1, j = lane & 1;
                bulk_g2s(ring + sl * SB + (2 * gg + j) * CP * TB,
                         a.img + ((size_t)tile_of(4 * r.q + gg, j) * a.C + r.c) * TB, unsigned(nc * TB), &full[sl]);
            }
        };
        auto issue_x = [&](const Rd &r, int sl) {   // the activations of round r (valid k-steps only)
            const int nc = r.ce - r.c < CP ? r.ce - r.c : CP;
            const int kb = K16 - 4 * r.c;
            const unsigned ng16 = unsigned(kb < 4 * nc ? kb : 4 * nc);   // 16-input groups of the round
            if (lane == 0) mbar_expect(&full[sl], MT * 512u * ng16 + 64u * ng16);
            __syncwarp();
            uint8_t *base = ring + sl * SB + WB;
            if (lane < MT)   // row block `lane`: its groups are one run of the operand format
                bulk_g2s(base + lane * XB, a.xf + act_group(a.K, a.x_row0 + 8 * lane, 4 * r.c), 512u * ng16, &full[sl]);
            else if (lane == MT)
                bulk_g2s(base + MT * XB, a.xs + (size_t)(4 * r.c) * kMaxRows, 64u * ng16, &full[sl]);
        };
        // a round whose copies are not issued (the pass failed before this launch): two plain arrivals
        // complete its phase without data, so no wait of the compute warps runs out
        auto arrive_only = [&](int sl, int n) {
            if (lane == 0)
                for (int i = 0; i < n; ++i) mbar_arrive(&full[sl]);
            __syncwarp();
        };
        Rd r;
        rd_at_quad(r, int(u0 / a.C), int(u0 % a.C));
        const Rd r0 = r;
        int k = 0;
        if (!a.stall) {
            // weights are immutable: the first rounds' weights go out before the previous kernel ends
            for (; k < S && rd_valid(r); ++k, rd_next(r)) issue_w(r, k);
        }
        pdl_wait();
        pdl_trigger();
        // The pass this launch belongs to may have failed already: then no more copies are issued and the
        // rounds complete empty. The flag's load is in flight while the prefetched rounds' activations go
        // out (those copies are harmless either way).
        const int errv = (a.skip_on_err && a.err) ? *reinterpret_cast<volatile int *>(a.err) : 0;
        {
            Rd rx = r0;
            for (int k2 = 0; k2 < k; ++k2, rd_next(rx)) issue_x(rx, k2);
        }
        const bool skip = errv != 0;
        if (!a.stall || skip) {
            for (; rd_valid(r); ++k, rd_next(r)) {
                const int sl = k % S;
                // once any wait of the CTA has given up, nothing more is issued
                if (!mbar_wait(&empty[sl], unsigned(k / S - 1) & 1u, &s_bad) || s_bad) break;
                if (skip) {
                    arrive_only(sl, 2);
                } else {
                    issue_w(r, sl);
                    issue_x(r, sl);
                }
            }
        }
        if (lane == 0) s_issued = k;   // rounds whose copies went out (read after the final barrier)
    } else {
        // ---- compute warps ----
        const int gq = warp & 3, par = warp >> 2;
        pdl_wait();
        pdl_trigger();
        stamp_ready(a.ps);
        float acc[2][MT][4];
        auto zero = [&]() {
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int tt = 0; tt < MT; ++tt) acc[j][tt][0] = acc[j][tt][1] = acc[j][tt][2] = acc[j][tt][3] = 0.f;
        };
        zero();
        // per-lane offsets inside a slot (unit par; unit par + 4i is 4i chunks further)
        const int w_off = (2 * gq * CP + par) * TB;
        const int x_off = WB + 2048 * par + 64 * g + 16 * t;
        const int s_off = WB + MT * XB + 256 * par;
        Rd cr;
        rd_at_quad(cr, int(u0 / a.C), int(u0 % a.C));
        for (int k = 0; rd_valid(cr); ++k) {
            const int sl = k % S;
            // a round whose wait gave up is skipped (its slot may still be landing); the control flow,
            // and so every barrier of the compute warps, stays the same
            const bool landed = mbar_wait(&full[sl], unsigned(k / S) & 1u, &s_bad);
            const int ng = 4 * cr.q + gq;
            if (landed && ng < ngroups) {
                const uint8_t *slot = ring + sl * SB;
                if (FMT == W_Q41) {
                    int nblk[NU];
#pragma unroll
                    for (int i = 0; i < NU; ++i) {
                        const int c = cr.c + par + kGemmPar * i, kb = K16 - 4 * c;
                        nblk[i] = c < cr.ce ? (kb < 4 ? kb / 2 : 2) : 0;
                    }
                    // units in pairs (or one); live units are a prefix, so a pair past them is skipped whole
                    constexpr int NP = NU % 2 == 0 ? 2 : 1;
#pragma unroll
                    for (int i0 = 0; i0 < NU; i0 += NP) {
                        int np[NP];
#pragma unroll
                        for (int i = 0; i < NP; ++i) np[i] = nblk[i0 + i];
                        if (np[0] > 0)
                            q41_units<FMT, MT, NP>(acc, slot, w_off + kGemmPar * i0 * TB, x_off + 2048 * kGemmPar * i0,
                                                   s_off + 256 * kGemmPar * i0, np, lane);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < NU; ++i) {
                        const int c = cr.c + par + kGemmPar * i, kb = K16 - 4 * c;
                        if (c < cr.ce)
                            bf16_unit<FMT, MT>(acc, slot, w_off + kGemmPar * i * TB, x_off + 2048 * kGemmPar * i,
                                               kb < 4 ? kb : 4, lane);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sl]);   // this warp is done with the slot
            Rd nx = cr;
            rd_next(nx);
            if (nx.q != cr.q || !rd_valid(nx)) {
                // end of the quad's range in this CTA: add the four parities
                const int q = cr.q;
                float *mine = red + (par * 4 + gq) * (R * 32);
#pragma unroll
                for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int tok = 8 * tt + 2 * t + (i & 1), r = g + 8 * (i >> 1);
                        mine[tok * 32 + r] = acc[0][tt][i];
                        mine[tok * 32 + 16 + r] = acc[1][tt][i];
                    }
                compute_sync();
                const long qa = (long)q * a.C;
                const int first = int(cta_of(qa, U, G)), last = int(cta_of(qa + a.C - 1, U, G));
                const int nseg = last - first + 1, seg = blockIdx.x - first;
                constexpr int G4 = R * 32 / 4;   // one group's float4s
                float4 *red4 = reinterpret_cast<float4 *>(red);
                auto sum_par = [&](int gg, int e) {   // parities added in order
                    float4 v = red4[gg * G4 + e];
#pragma unroll
                    for (int pp = 1; pp < kGemmPar; ++pp) {
                        const float4 w = red4[(pp * 4 + gg) * G4 + e];
                        v.x += w.x, v.y += w.y, v.z += w.z, v.w += w.w;
                    }
                    return v;
                };
                if (EPI == EPI_PART || EPI == EPI_ROWS || EPI == EPI_QK) {
                    // the partial of every quad, the consumer (or the row step below) adds the segments
                    for (int te = threadIdx.x; te < 4 * G4; te += kGemmThreads) {
                        const int gg = te / G4, e = te % G4;
                        if (4 * q + gg < ngroups)
                            reinterpret_cast<float4 *>(a.part)[((size_t)(4 * q + gg) * a.maxseg + seg) * (kMaxRows * 8) + e] =
                                sum_par(gg, e);
                    }
                } else if (nseg > 1) {
                    // this CTA's partial of the quad: 4 groups x R rows x 32 columns, summed over parities
                    for (int te = threadIdx.x; te < 4 * G4; te += kGemmThreads) {
                        const int gg = te / G4, e = te % G4;
                        if (4 * q + gg < ngroups)
                            reinterpret_cast<float4 *>(a.part)[((size_t)(4 * q + gg) * a.maxseg + seg) * (kMaxRows * 8) + e] =
                                sum_par(gg, e);
                    }
                    // one thread publishes the CTA's partial (barrier, then fence and ticket)
                    compute_sync();
                    if (threadIdx.x == 0) {
                        __threadfence();
                        const int last_one = atomicAdd(a.cnt + q, 1) == nseg - 1;
                        if (last_one) __threadfence();
                        s_last = last_one;
                    }
                    compute_sync();
                    if (s_last) {
                        // every thread adds its float4 over the segments, in segment order
                        for (int te = threadIdx.x; te < 4 * G4; te += kGemmThreads) {
                            const int gg = te / G4, e = te % G4;
                            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (4 * q + gg < ngroups) {
                                const float4 *pp = reinterpret_cast<const float4 *>(a.part) +
                                                   (size_t)(4 * q + gg) * a.maxseg * (kMaxRows * 8) + e;
                                float4 l[8];
                                for (int s0 = 0; s0 < nseg; s0 += 8) {
#pragma unroll
                                    for (int s2 = 0; s2 < 8; ++s2)
                                        l[s2] = s0 + s2 < nseg ? __ldcg(pp + (s0 + s2) * (kMaxRows * 8)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                                    for (int s2 = 0; s2 < 8; ++s2)
                                        if (s0 + s2 < nseg) v.x += l[s2].x, v.y += l[s2].y, v.z += l[s2].z, v.w += l[s2].w;
                                }
                            }
                            red4[gg * G4 + e] = v;
                        }
                        if (threadIdx.x == 0) a.cnt[q] = 0;
                    }
                    compute_sync();
                } else {
                    constexpr int PER = (4 * G4 + kGemmThreads - 1) / kGemmThreads;
                    float4 v[PER];
#pragma unroll
                    for (int i = 0; i < PER; ++i) {
                        const int te = threadIdx.x + i * kGemmThreads;
                        if (te < 4 * G4) v[i] = sum_par(te / G4, te % G4);
                    }
                    compute_sync();
#pragma unroll
                    for (int i = 0; i < PER; ++i) {
                        const int te = threadIdx.x + i * kGemmThreads;
                        if (te < 4 * G4) red4[te] = v[i];
                    }
                    compute_sync();
                }
                const bool fin = EPI != EPI_PART && EPI != EPI_ROWS && EPI != EPI_QK && (nseg == 1 || s_last);
                const int ngq = 4 * q + gq;
                if (fin && par == 0 && ngq < ngroups) {
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int tok = 8 * tt + 2 * t + (i & 1), r = g + 8 * (i >> 1);
                            acc[0][tt][i] = red[gq * (R * 32) + tok * 32 + r];
                            acc[1][tt][i] = red[gq * (R * 32) + tok * 32 + 16 + r];
                        }
                    epilogue<MT, EPI>(a, acc, tile_of(ngq, 0), tile_of(ngq, 1), ngq, lane);
                }
                compute_sync();   // red and s_last are reused by the next quad
                zero();
                if (threadIdx.x == 0) s_last = 0;
            }
            cr = nx;
        }
    }
    __syncthreads();   // every warp is done
    if (EPI == EPI_ROWS || EPI == EPI_QK) {
        // The steps that need whole rows of the product, by the last CTAs to finish: each CTA takes a
        // ticket once its partials are out; a worker waits (bounded) until every CTA has taken one, then
        // adds the segments it needs and applies its steps. EPI_ROWS: one row per worker (the row step);
        // EPI_QK: one (row, head) per warp (the q/k steps). Every CTA of the grid is resident (one per
        // SM, and no later kernel starts before all of them have), so the wait always ends.
        __shared__ float red[33];
        __shared__ float4 red4[33];
        constexpr int kWarps = kGemmBlock / 32;
        int tasks0 = 0, total = a.M;
        if (EPI == EPI_QK) {
            tasks0 = a.qk[0].M * qk_heads(a.qk[0]);
            total = tasks0 + (a.nqk > 1 ? a.qk[1].M * qk_heads(a.qk[1]) : 0);
        }
        const int want = EPI == EPI_ROWS ? total : (total + kWarps - 1) / kWarps;
        const int nw = G < want ? G : want;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_ticket = atomicAdd(a.row_cnt, 1);
        __syncthreads();
        const int w = s_ticket - (G - nw);
        if (w >= 0) {
            constexpr int PER = kProductRowPer;
            float4 wp[PER], wn[PER];
            if (EPI == EPI_ROWS) row_weights<PER>(a.row, wp, wn);   // in flight during the wait below
            if (threadIdx.x == 0) {
                const unsigned long long t0 = globaltimer_ns();
                for (;;) {
                    int seen;
                    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(a.row_cnt) : "memory");
                    if (seen >= G) break;
                    if (globaltimer_ns() - t0 > kWaitLimitNs) {
                        s_bad = 1;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            __syncthreads();
            if (!s_bad) {
                if (EPI == EPI_ROWS) {
                    for (int m = w; m < a.M; m += nw) row_step<PER>(a.row, m, wp, wn, red, red4);
                } else {
                    for (int t = w * kWarps + warp; t < total; t += nw * kWarps) {
                        const int which = t < tasks0 ? 0 : 1, tt = which ? t - tasks0 : t;
                        const int heads = qk_heads(a.qk[which]);
                        qk_task(a.qk[which], tt / heads, tt % heads, lane);
                    }
                }
            }
            __syncthreads();
            if (threadIdx.x == 0 && atomicAdd(a.row_cnt + 1, 1) == nw - 1) {
                a.row_cnt[0] = 0;   // every CTA has arrived and every worker is done
                a.row_cnt[1] = 0;
            }
        }
        __syncthreads();
    }
    if (s_bad) {
        // A wait gave up: copies issued into a slot may still be in flight. Before the CTA exits, wait
        // (bounded again) for the last round issued into each slot; its phase completes only once
        // every byte of it, and of the rounds before it in that slot, has landed.
        if (warp == kGemmWarps && lane == 0) {
            const int issued = s_issued;
            volatile int drain_bad = 0;
            for (int sl = 0; sl < S && sl < issued; ++sl) {
                const int last = sl + (issued - 1 - sl) / S * S;
                mbar_wait(&full[sl], unsigned(last / S) & 1u, &drain_bad);
                drain_bad = 0;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, kErrWaitTimeout);
    }
    stamp_done(a.ps);
}

// ---------------------------------------------------------------------------------------------------
// bf16 head: logits of M rows over the vocabulary, fused with the first-maximum argmax and, for a
// verify, the longest-prefix acceptance.
// ---------------------------------------------------------------------------------------------------
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

constexpr int kHeadPad = 64;   // bytes added per staged row: conflict-free 16-byte fragment reads

template <int MT>
__global__ void __launch_bounds__(kWarpsPerCta * 32) k_head(GemmArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float wval[kWarpsPerCta][kMaxRows];
    __shared__ int widx[kWarpsPerCta][kMaxRows];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int rowb = a.K * 4 + kHeadPad;
    const int K16 = a.K / 16;

    const int ntiles = a.N / 16;
    const int gw = blockIdx.x * kWarpsPerCta + warp, nw = gridDim.x * kWarpsPerCta;
    const int t0 = int((long)gw * ntiles / nw), t1 = int((long)(gw + 1) * ntiles / nw);
    float bv[MT][2];
    int bi[MT][2];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) bv[tt][0] = bv[tt][1] = -INFINITY, bi[tt][0] = bi[tt][1] = 0x7fffffff;

    // work units: pairs of tiles (the last may be single) x chunks, streamed with P units in flight
    const int npairs = (t1 - t0 + 1) / 2;
    const int units = npairs * a.C;
    constexpr int P = 2;
    uint4 w[P][2][4];
    auto tile_of = [&](int pr, int j) { return t0 + 2 * pr + j; };
    auto load = [&](int u, uint4 (&dst)[2][4]) {
        const int pr = u / a.C, c = u % a.C;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int tl = tile_of(pr, j);
            const int tv = tl < t1 ? tl : t1 - 1;   // a single last tile reloads itself (result unused)
            const uint8_t *b = a.img + ((size_t)tv * a.C + c) * 2048;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) dst[j][ks] = ldg_stream(b + 512 * ks + 16 * lane);
        }
    };
#pragma unroll
    for (int p = 0; p < P; ++p)
        if (p < units) load(p, w[p]);
    pdl_wait();
    pdl_trigger();
    stamp_ready(a.ps);
    // stage the activation fragments of all rows (one asynchronous copy round trip)
    for (int e = threadIdx.x; e < MT * 8 * K16 * 4; e += blockDim.x) {
        const int tok = e / (K16 * 4), rest = e % (K16 * 4);
        uint8_t *dst = smem + tok * rowb + rest * 16;
        if (tok < a.M)
            cp_async16(dst, a.xf + act_group(a.K, a.x_row0 + tok, rest >> 2) + (rest & 3) * 4);
        else
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_wait_all();
    __syncthreads();

    float acc[2][MT][4];
    for (int ub = 0; ub < units; ub += P) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int u = ub + p;
            if (u < units) {
                const int pr = u / a.C, c = u % a.C;
                if (c == 0) {
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int tt = 0; tt < MT; ++tt) acc[j][tt][0] = acc[j][tt][1] = acc[j][tt][2] = acc[j][tt][3] = 0.f;
                }
                const uint4 (&wv)[2][4] = w[p];
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint4 b[MT];
#pragma unroll
                    for (int tt = 0; tt < MT; ++tt)
                        b[tt] = *reinterpret_cast<const uint4 *>(smem + (8 * tt + g) * rowb + ((4 * c + ks) * 4 + t) * 16);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int tt = 0; tt < MT; ++tt)
                            mma_bf16(acc[j][tt], wv[j][ks].x, wv[j][ks].y, wv[j][ks].z, wv[j][ks].w, b[tt].x, b[tt].y);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int tt = 0; tt < MT; ++tt)
                            mma_bf16(acc[j][tt], wv[j][ks].x, wv[j][ks].y, wv[j][ks].z, wv[j][ks].w, b[tt].z, b[tt].w);
                }
                if (u + P < units) load(u + P, w[p]);
                if (c == a.C - 1) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int tl = tile_of(pr, j);
                        if (tl >= t1) continue;
#pragma unroll
                        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int tok = 8 * tt + 2 * t + (i & 1);
                                const int v = 16 * tl + g + 8 * (i >> 1);
                                const float val = acc[j][tt][i];
                                if (tok < a.M && a.logits) a.logits[(long)tok * a.ldl + v] = val;
                                if (better(val, v, bv[tt][i & 1], bi[tt][i & 1])) bv[tt][i & 1] = val, bi[tt][i & 1] = v;
                            }
                    }
                }
            }
        }
    }
    // reduce over lanes with the same t (same tokens)
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv[tt][h], o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi[tt][h], o);
                if (better(ov, oi, bv[tt][h], bi[tt][h])) bv[tt][h] = ov, bi[tt][h] = oi;
            }
            if (g == 0) {
                const int tok = 8 * tt + 2 * t + h;
                if (tok < kMaxRows) wval[warp][tok] = bv[tt][h], widx[warp][tok] = bi[tt][h];
            }
        }
    __syncthreads();
    if (threadIdx.x < a.M) {
        const int tok = threadIdx.x;
        float v = wval[0][tok];
        int i = widx[0][tok];
        for (int w2 = 1; w2 < kWarpsPerCta; ++w2)
            if (better(wval[w2][tok], widx[w2][tok], v, i)) v = wval[w2][tok], i = widx[w2][tok];
        a.am_val[(long)blockIdx.x * kMaxRows + tok] = v;
        a.am_idx[(long)blockIdx.x * kMaxRows + tok] = i;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.am_cnt, 1) == (int)gridDim.x - 1);
    __syncthreads();
    stamp_done(a.ps);
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < a.M) {
        const int tok = threadIdx.x;
        float v = -INFINITY;
        int i = 0x7fffffff;
        for (int b = 0; b < (int)gridDim.x; ++b) {
            const float bvv = __ldcg(a.am_val + (long)b * kMaxRows + tok);
            const int bii = __ldcg(a.am_idx + (long)b * kMaxRows + tok);
            if (better(bvv, bii, v, i)) v = bvv, i = bii;
        }
        if (a.am_dst == AM_VERIFY) a.st->target[tok] = i;
        else if (a.am_dst == AM_DRAFT) a.st->props[tok] = i;
        else a.am_out[tok] = i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (a.am_dst == AM_VERIFY) {
            // longest prefix: proposal rows[i] (position n+i) accepted while it equals target[i-1]
            int acc_len = 0;
            while (acc_len + 1 < a.M && a.st->rows[acc_len + 1] == a.st->target[acc_len]) ++acc_len;
            a.st->accepted = acc_len;
        }
        *a.am_cnt = 0;
    }
    stamp_done(a.ps);
}

// ---------------------------------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------------------------------
// Grid of a product: one CTA per SM at most, and at least four units (chunks of a quad) per CTA.
int gemm_grid(int C, int N) {
    const long Q = (N / 32 + 3) / 4;
    const long U = Q * C;
    long G = 152;
    if (G > U / 4) G = U / 4;
    return int(G < 1 ? 1 : G);
}

int gemm_maxseg(int C, int N) {
    const int G = gemm_grid(C, N);
    const long Q = (N / 32 + 3) / 4;
    const long U = Q * C;
    int mx = 1;
    for (long q = 0; q < Q; ++q) {
        const long a0 = ((q * C + 1) * G - 1) / U, a1 = ((q * C + C) * G - 1) / U;
        mx = std::max(mx, int(a1 - a0 + 1));
    }
    return mx;
}

size_t gemm_scratch_floats(int C, int N) {
    const int ms = gemm_maxseg(C, N);
    return ms > 1 ? (size_t)(N / 32) * ms * kMaxRows * 32 : 0;
}

size_t gemm_part_floats(int C, int N) { return (size_t)(N / 32) * gemm_maxseg(C, N) * kMaxRows * 32; }

// dynamic shared memory of a product: the parity reduction buffer and the ring
template <int FMT, int MT, int EPI>
static cudaError_t run_gemm(const GemmArgs &a, cudaStream_t s) {
    if (a.x_row0 % 8) return cudaErrorInvalidValue;   // products read whole row blocks
    constexpr int smem = red_bytes<MT>() + ring_slots<FMT, MT>() * slot_bytes<FMT, MT>();
    static_assert(smem <= kGemmSmemBudget, "product shared memory");
    static bool attr[kMaxDevices] = {};
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (!attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm<FMT, MT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    return launch_pdl(k_gemm<FMT, MT, EPI>, dim3(gemm_grid(a.C, a.N)), dim3(kGemmBlock), (size_t)smem, s, a);
}

size_t head_smem(int K, int MT) { return (size_t)MT * 8 * (K * 4 + kHeadPad); }

int head_grid(int C, int M, int N) {
    const int MT = M > 8 ? 2 : 1;
    const size_t smem = head_smem(C * 64, MT);
    const int per_sm = smem <= 48 * 1024 ? 4 : (smem <= 100 * 1024 ? 2 : 1);
    int grid = 152 * per_sm;
    const int ntiles = N / 16;
    if (grid * kWarpsPerCta > ntiles) grid = (ntiles + kWarpsPerCta - 1) / kWarpsPerCta;
    return grid;
}

template <int MT>
static cudaError_t run_head(const GemmArgs &a, cudaStream_t s) {
    const size_t smem = head_smem(a.K, MT);
    static bool attr[kMaxDevices] = {};
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (!attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_head<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    return launch_pdl(k_head<MT>, dim3(head_grid(a.C, a.M, a.N)), dim3(kWarpsPerCta * 32), smem, s, a);
}

cudaError_t launch_gemm(int fmt, int epi, const GemmArgs &a, cudaStream_t s) {
    const bool two = a.M > 8;
    if (epi == EPI_ARGMAX) return two ? run_head<2>(a, s) : run_head<1>(a, s);
#define DFL_GEMM_CASE(F, E) \
    if (fmt == F && epi == E) return two ? run_gemm<F, 2, E>(a, s) : run_gemm<F, 1, E>(a, s);
    DFL_GEMM_CASE(W_Q41, EPI_F32)
    DFL_GEMM_CASE(W_Q41, EPI_PART)
    DFL_GEMM_CASE(W_Q41, EPI_ROWS)
    DFL_GEMM_CASE(W_Q41, EPI_QK)
    DFL_GEMM_CASE(W_Q41, EPI_GLU)
    DFL_GEMM_CASE(W_Q41, EPI_SILU_MUL)
    DFL_GEMM_CASE(W_BF16, EPI_F32)
#undef DFL_GEMM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace dfl
