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

namespace dfl {

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
    pdl_wait();
    pdl_trigger();
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
// activation staging: the chunks a CTA needs are copied to shared memory once (one asynchronous copy
// round trip), so the unit loop reads its B fragments and sums from shared memory.
// Per slot (one 64-input chunk): sums [4 groups][16 rows] fp32 (256 B), then R = 8*MT rows of 256 B
// fragments; inside a row the four 64-byte k-steps are stored at position ks ^ (row & 1), so the two
// rows a quarter warp reads fall on different banks.
// ---------------------------------------------------------------------------------------------------
template <int MT>
__host__ __device__ constexpr int slot_bytes() { return 256 + MT * 8 * 256; }
template <int MT>
__host__ __device__ constexpr int red_bytes() { return 16 * MT * 8 * 32 * 4; }   // [4 parities][4 groups][R][32]

// copy the chunks of units [s0, s1) (at most `slots` distinct chunks; slot of chunk c = (c - s0 % C) mod C)
template <int MT>
__device__ __forceinline__ void stage_x(const GemmArgs &a, uint8_t *xs_sm, long s0, long s1) {
    constexpr int R = MT * 8;
    const int K16 = a.K / 16;
    const long span = s1 - s0;
    const int nch = int(span < a.C ? span : a.C);
    const int cb = int(s0 % a.C);
    const int per = 16 + R * 16;   // 16-byte pieces per slot
    for (int e = threadIdx.x; e < nch * per; e += blockDim.x) {
        const int slot = e / per, r = e % per;
        const int c = (cb + slot) % a.C;
        uint8_t *base = xs_sm + slot * slot_bytes<MT>();
        if (r < 16) {   // sums: group 4c + r/4, rows 4*(r%4) .. +3
            const int kb = 4 * c + (r >> 2);
            uint8_t *dst = base + 16 * r;
            if (kb < K16) cp_async16(dst, a.xs + kb * kMaxRows + 4 * (r & 3));
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        } else {
            const int rr = r - 16, tok = rr >> 4, ks = (rr >> 2) & 3, t = rr & 3;
            const int kb = 4 * c + ks;
            uint8_t *dst = base + 256 + tok * 256 + ((ks ^ (tok & 1)) * 4 + t) * 16;
            if (kb < K16)
                cp_async16(dst, a.xf + (((long)(a.x_row0 + tok) * K16 + kb) * 4 + t) * 4);
            else
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    cp_async_wait_all();
}

// B fragment (hi in .x/.y, lo in .z/.w) of k-step ks for rows 8*tt + g
__device__ __forceinline__ uint4 frag(const uint8_t *slot, int tt, int ks, int g, int t) {
    const int tok = 8 * tt + g;
    return *reinterpret_cast<const uint4 *>(slot + 256 + tok * 256 + ((ks ^ (tok & 1)) * 4 + t) * 16);
}

// ---------------------------------------------------------------------------------------------------
// one unit of work: a 64-input chunk of two 16-column tiles
// ---------------------------------------------------------------------------------------------------
// Q4_1: the codes enter the tensor cores as 128 + q (exact in bf16), so per 32-block b
//   sum_k x_k w_k = d_b sum_k x_k (128 + q_k) + (m_b - 128 d_b) sum_k x_k,
// with sum_k x_k the staged per-16 sums of the operand (hi + lo) values.
template <int MT>
__device__ __forceinline__ void q41_unit(float (&acc)[2][MT][4], const uint4 (&nb)[2], const uint4 (&sc)[2],
                                         const uint8_t *slot, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const float *sums = reinterpret_cast<const float *>(slot);
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        float2 S[MT];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
            const float2 s0 = *reinterpret_cast<const float2 *>(sums + (2 * blk) * kMaxRows + 8 * tt + 2 * t);
            const float2 s1 = *reinterpret_cast<const float2 *>(sums + (2 * blk + 1) * kMaxRows + 8 * tt + 2 * t);
            S[tt] = make_float2(s0.x + s1.x, s0.y + s1.y);
        }
        float ch[2][MT][4], cl[2][MT][4];   // hi and lo chains
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) ch[j][tt][i] = cl[j][tt][i] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int ks = 2 * blk + kk;
            uint4 b[MT];
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) b[tt] = frag(slot, tt, ks, g, t);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t w = ks == 0 ? nb[j].x : ks == 1 ? nb[j].y : ks == 2 ? nb[j].z : nb[j].w;
                const uint32_t a0 = nib_pair_bf16(w), a1 = nib_pair_bf16(w >> 4);
                const uint32_t a2 = nib_pair_bf16(w >> 8), a3 = nib_pair_bf16(w >> 12);
#pragma unroll
                for (int tt = 0; tt < MT; ++tt) {
                    mma_bf16(ch[j][tt], a0, a1, a2, a3, b[tt].x, b[tt].y);
                    mma_bf16(cl[j][tt], a0, a1, a2, a3, b[tt].z, b[tt].w);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t dlo = blk ? sc[j].z : sc[j].x, dhi = blk ? sc[j].w : sc[j].y;
            const float2 flo = __half22float2(*reinterpret_cast<__half2 *>(&dlo));   // (d, m) of column g
            const float2 fhi = __half22float2(*reinterpret_cast<__half2 *>(&dhi));   // column g + 8
            const float mlo = fmaf(-128.f, flo.x, flo.y), mhi = fmaf(-128.f, fhi.x, fhi.y);
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
                acc[j][tt][0] = fmaf(mlo, S[tt].x, fmaf(flo.x, ch[j][tt][0] + cl[j][tt][0], acc[j][tt][0]));
                acc[j][tt][1] = fmaf(mlo, S[tt].y, fmaf(flo.x, ch[j][tt][1] + cl[j][tt][1], acc[j][tt][1]));
                acc[j][tt][2] = fmaf(mhi, S[tt].x, fmaf(fhi.x, ch[j][tt][2] + cl[j][tt][2], acc[j][tt][2]));
                acc[j][tt][3] = fmaf(mhi, S[tt].y, fmaf(fhi.x, ch[j][tt][3] + cl[j][tt][3], acc[j][tt][3]));
            }
        }
    }
}

template <int MT>
__device__ __forceinline__ void bf16_unit(float (&acc)[2][MT][4], const uint4 (&w)[2][4], const uint8_t *slot, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint4 b[MT];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) b[tt] = frag(slot, tt, ks, g, t);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
                mma_bf16(acc[j][tt], w[j][ks].x, w[j][ks].y, w[j][ks].z, w[j][ks].w, b[tt].x, b[tt].y);
                mma_bf16(acc[j][tt], w[j][ks].x, w[j][ks].y, w[j][ks].z, w[j][ks].w, b[tt].z, b[tt].w);
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
// One CTA per SM, 16 warps: warp w takes column group gq = w % 4 of the current quad and chunk parity
// par = w / 4, i.e. chunks c with c % 4 == par of the CTA's chunk range of that quad. At the end of a
// range the four parities are added in shared memory (order 0..3); a quad split over several CTAs
// leaves one partial per CTA, added by the last CTA to finish it (order of the segments).
// The CTA's unit range [u0, u1) is cut into stages of at most a.slots distinct chunks (one stage
// unless the range is long); each stage's activations are staged in shared memory, and the loop walks
// the pieces (quad sub-range x stage) in order.
constexpr int kGemmWarps = 16;

__device__ __forceinline__ long cta_of(long u, long U, int G) { return ((u + 1) * G - 1) / U; }

template <int FMT, int MT, int EPI>
__global__ void __launch_bounds__(kGemmWarps * 32, 1) k_gemm(GemmArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_last;
    constexpr int R = MT * 8;
    float *red = reinterpret_cast<float *>(smem);               // [4 par][4 gq][R][32]
    uint8_t *xs_sm = smem + red_bytes<MT>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int gq = warp & 3, par = warp >> 2;
    const int ngroups = a.N / 32;
    const int Q = (ngroups + 3) / 4;
    const long U = (long)Q * a.C;
    const int G = gridDim.x;
    const long u0 = (long)blockIdx.x * U / G, u1 = (long)(blockIdx.x + 1) * U / G;
    constexpr int P = (FMT == W_Q41 && MT == 1) ? 4 : 2;
    constexpr int TB = FMT == W_Q41 ? 640 : 2048;
    // stage length in units: the whole range when its distinct chunks fit
    const long span = u1 - u0;
    const long L = (span < a.C ? span : a.C) <= a.slots ? span : a.slots;
    auto stage_end = [&](long x) -> long {
        const long e = u0 + ((x - u0) / L + 1) * L;
        return e < u1 ? e : u1;
    };
    auto piece_end = [&](long x) -> long {
        const long qe = (x / a.C + 1) * a.C;
        const long se = stage_end(x);
        return qe < se ? qe : se;
    };

    auto tiles = [&](int q, int &nt0, int &nt1, int &ng) {
        ng = 4 * q + gq;
        const int ngc = ng < ngroups ? ng : ngroups - 1;   // an idle warp of the last quad reads valid memory
        nt0 = (EPI == EPI_GLU) ? ngc : 2 * ngc;
        nt1 = (EPI == EPI_GLU) ? ngc + ngroups : 2 * ngc + 1;
    };
    uint4 nb[P][2], sc[P][2];
    uint4 w[P][2][4];
    auto load = [&](int q, int c, int p) {
        int nt0, nt1, ng;
        tiles(q, nt0, nt1, ng);
        const uint8_t *b0 = a.img + ((size_t)nt0 * a.C + c) * TB;
        const uint8_t *b1 = a.img + ((size_t)nt1 * a.C + c) * TB;
        if (FMT == W_Q41) {
            nb[p][0] = ldg_stream(b0 + 16 * lane);
            nb[p][1] = ldg_stream(b1 + 16 * lane);
            sc[p][0] = ldg_stream(b0 + 512 + 16 * g);
            sc[p][1] = ldg_stream(b1 + 512 + 16 * g);
        } else {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                w[p][0][ks] = ldg_stream(b0 + 512 * ks + 16 * lane);
                w[p][1][ks] = ldg_stream(b1 + 512 * ks + 16 * lane);
            }
        }
    };
    // this warp's first chunk of a piece starting at unit ps (chunks c % 4 == par)
    auto my_first = [&](long ps) -> int { const int ca = int(ps % a.C); return ca + ((par - ca) % 4 + 4) % 4; };
    auto prefetch = [&](long ps) {   // the first P units of the piece starting at ps
        if (ps >= u1) return;
        const int q = int(ps / a.C);
        const int ce = int(piece_end(ps) - (long)q * a.C);
        const int c0 = my_first(ps);
#pragma unroll
        for (int p = 0; p < P; ++p)
            if (c0 + 4 * p < ce) load(q, c0 + 4 * p, p);
    };
    // weights are immutable: the first loads are issued before the previous kernel has finished
    prefetch(u0);
    pdl_wait();
    pdl_trigger();

    long s0 = u0, s1 = stage_end(u0);
    stage_x<MT>(a, xs_sm, s0, s1);
    __syncthreads();

    float acc[2][MT][4];
    auto zero = [&]() {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) acc[j][tt][0] = acc[j][tt][1] = acc[j][tt][2] = acc[j][tt][3] = 0.f;
    };
    zero();
    for (long ps = u0; ps < u1;) {
        const int q = int(ps / a.C);
        const long pe = piece_end(ps);
        const long qend = ((long)q + 1) * a.C < u1 ? ((long)q + 1) * a.C : u1;
        const int ce = int(pe - (long)q * a.C);
        const int c0 = my_first(ps);
        const int cbase = int(s0 % a.C);
        const int nmine = c0 < ce ? (ce - c0 + 3) / 4 : 0;
        for (int ib = 0; ib < nmine; ib += P) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int i = ib + p;
                if (i < nmine) {
                    const int c = c0 + 4 * i;
                    const uint8_t *slot = xs_sm + ((c - cbase + a.C) % a.C) * slot_bytes<MT>();
                    if (FMT == W_Q41) q41_unit<MT>(acc, nb[p], sc[p], slot, lane);
                    else bf16_unit<MT>(acc, w[p], slot, lane);
                    if (i + P < nmine) load(q, c + 4 * P, p);
                }
            }
        }
        // the next piece's first weights stream while this one is reduced or restaged
        prefetch(pe);
        if (pe == qend) {
            // add the four parities
            float *mine = red + (par * 4 + gq) * (R * 32);
#pragma unroll
            for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = 8 * tt + 2 * t + (i & 1), r = g + 8 * (i >> 1);
                    mine[tok * 32 + r] = acc[0][tt][i];
                    mine[tok * 32 + 16 + r] = acc[1][tt][i];
                }
            __syncthreads();
            const long qa = (long)q * a.C;
            const int first = int(cta_of(qa, U, G)), last = int(cta_of(qa + a.C - 1, U, G));
            const int nseg = last - first + 1, seg = blockIdx.x - first;
            const int ng = 4 * q + gq;
            constexpr int GR = R * 32;   // one group's elements
            auto red_at = [&](int pp, int gg, int rc) -> float & { return red[(pp * 4 + gg) * GR + rc]; };
            if (nseg > 1) {
                // this CTA's partial of the quad: 4 groups x R rows x 32 columns, summed over parities
                for (int e = threadIdx.x; e < 4 * GR; e += blockDim.x) {
                    const int gg = e / GR, rc = e % GR;
                    if (4 * q + gg < ngroups) {
                        const float v = ((red_at(0, gg, rc) + red_at(1, gg, rc)) + red_at(2, gg, rc)) + red_at(3, gg, rc);
                        a.part[((size_t)(4 * q + gg) * a.maxseg + seg) * (kMaxRows * 32) + rc] = v;
                    }
                }
                // one thread publishes the CTA's partial (barrier, then fence and ticket)
                __syncthreads();
                if (threadIdx.x == 0) {
                    __threadfence();
                    const int last_one = atomicAdd(a.cnt + q, 1) == nseg - 1;
                    if (last_one) __threadfence();
                    s_last = last_one;
                }
                __syncthreads();
                if (s_last) {
                    // every thread adds its elements over the segments, in segment order
                    for (int e = threadIdx.x; e < 4 * GR; e += blockDim.x) {
                        const int gg = e / GR, rc = e % GR;
                        float v = 0.f;
                        if (4 * q + gg < ngroups) {
                            const float *pp = a.part + (size_t)(4 * q + gg) * a.maxseg * (kMaxRows * 32) + rc;
                            float l[16];
#pragma unroll
                            for (int s2 = 0; s2 < 16; ++s2) l[s2] = s2 < nseg ? __ldcg(pp + s2 * (kMaxRows * 32)) : 0.f;
                            for (int s2 = 0; s2 < nseg && s2 < 16; ++s2) v += l[s2];
                            for (int s2 = 16; s2 < nseg; ++s2) v += __ldcg(pp + s2 * (kMaxRows * 32));
                        }
                        red_at(0, gg, rc) = v;
                    }
                    if (threadIdx.x == 0) a.cnt[q] = 0;
                }
                __syncthreads();
            } else {
                for (int e = threadIdx.x; e < 4 * GR; e += blockDim.x) {
                    const int gg = e / GR, rc = e % GR;
                    red_at(0, gg, rc) = ((red_at(0, gg, rc) + red_at(1, gg, rc)) + red_at(2, gg, rc)) + red_at(3, gg, rc);
                }
                __syncthreads();
            }
            const bool fin = nseg == 1 || s_last;
            if (fin && par == 0 && ng < ngroups) {
#pragma unroll
                for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int tok = 8 * tt + 2 * t + (i & 1), r = g + 8 * (i >> 1);
                        acc[0][tt][i] = red_at(0, gq, tok * 32 + r);
                        acc[1][tt][i] = red_at(0, gq, tok * 32 + 16 + r);
                    }
                int nt0, nt1, ngx;
                tiles(q, nt0, nt1, ngx);
                epilogue<MT, EPI>(a, acc, nt0, nt1, ng, lane);
            }
            __syncthreads();   // red is reused by the next quad
            zero();
            if (threadIdx.x == 0) s_last = 0;
        }
        if (pe == s1 && pe < u1) {   // next stage
            __syncthreads();         // every warp is done with the staged activations
            s0 = s1;
            s1 = stage_end(s0);
            stage_x<MT>(a, xs_sm, s0, s1);
            __syncthreads();
        }
        ps = pe;
    }
}

// ---------------------------------------------------------------------------------------------------
// bf16 head: logits of M rows over the vocabulary, fused with the first-maximum argmax and, for a
// verify, the longest-prefix acceptance.
// ---------------------------------------------------------------------------------------------------
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

constexpr int kHeadPad = 64;   // bytes added per staged row: conflict-free 16-byte fragment reads

template <int MT>
__global__ void __launch_bounds__(128) k_head(GemmArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
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
    // stage the activation fragments of all rows (one asynchronous copy round trip)
    for (int e = threadIdx.x; e < MT * 8 * K16 * 4; e += blockDim.x) {
        const int tok = e / (K16 * 4), rest = e % (K16 * 4);
        uint8_t *dst = smem + tok * rowb + rest * 16;
        if (tok < a.M)
            cp_async16(dst, reinterpret_cast<const uint8_t *>(a.xf) + ((long)(a.x_row0 + tok) * K16 * 4 + rest) * 16);
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
                        for (int tt = 0; tt < MT; ++tt) {
                            mma_bf16(acc[j][tt], wv[j][ks].x, wv[j][ks].y, wv[j][ks].z, wv[j][ks].w, b[tt].x, b[tt].y);
                            mma_bf16(acc[j][tt], wv[j][ks].x, wv[j][ks].y, wv[j][ks].z, wv[j][ks].w, b[tt].z, b[tt].w);
                        }
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
        else a.st->props[tok] = i;
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

// dynamic shared memory of a product: the parity reduction buffer and the activation slots
constexpr int kGemmSmemBudget = 224 * 1024;

template <int FMT, int MT, int EPI>
static cudaError_t run_gemm(const GemmArgs &a0, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm<FMT, MT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kGemmSmemBudget);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    GemmArgs a = a0;
    const int G = gemm_grid(a.C, a.N);
    const long U = (long)((a.N / 32 + 3) / 4) * a.C;
    const long per_cta = (U + G - 1) / G;
    const int most = (kGemmSmemBudget - red_bytes<MT>()) / slot_bytes<MT>();
    const long need = per_cta < a.C ? per_cta : a.C;
    a.slots = int(need < most ? need : most);
    const size_t smem = (size_t)red_bytes<MT>() + (size_t)a.slots * slot_bytes<MT>();
    return launch_pdl(k_gemm<FMT, MT, EPI>, dim3(G), dim3(kGemmWarps * 32), smem, s, a);
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
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_head<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch_pdl(k_head<MT>, dim3(head_grid(a.C, a.M, a.N)), dim3(128), smem, s, a);
}

cudaError_t launch_gemm(int fmt, int epi, const GemmArgs &a, cudaStream_t s) {
    const bool two = a.M > 8;
    if (epi == EPI_ARGMAX) return two ? run_head<2>(a, s) : run_head<1>(a, s);
#define DFL_GEMM_CASE(F, E) \
    if (fmt == F && epi == E) return two ? run_gemm<F, 2, E>(a, s) : run_gemm<F, 1, E>(a, s);
    DFL_GEMM_CASE(W_Q41, EPI_F32)
    DFL_GEMM_CASE(W_Q41, EPI_GLU)
    DFL_GEMM_CASE(W_Q41, EPI_SILU_MUL)
    DFL_GEMM_CASE(W_BF16, EPI_F32)
#undef DFL_GEMM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace dfl
