// gemm.cu -- the skinny products of the step (M = 1..16 rows).
//
// Every projection of the batched verify and of the draft is one M-row product over a weight image
// streamed once from HBM (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass",
// "What changes": a verify of k rows used to cost k passes over the weights). Weights are Q4_1
// (model card "Nemotron-3.5-Bolt-E4B-DFlash-NPU2", spec table: "5 bits per weight with scales and
// minimums") except fc and the head, which are bf16.
//
// Layout. A weight matrix of K inputs x N outputs is cut into tiles of 16 output columns x 64 inputs.
// Tile (nt, c) of a matrix with C = ceil(K/64) chunks sits at offset (nt*C + c) * tile_bytes, so one
// column strip's whole K range is contiguous. Inside a tile the data is ordered by the lane of the
// warp that consumes it as the A operand of mma.m16n8k16 (rows = output columns, columns = inputs):
//   Q4_1 (640 B): lane L = 4g + t holds 16 B of codes at 16L: word s (k-step s, inputs 16s..16s+15)
//     packs, low to high nibble, q(g,2t) q(g+8,2t) q(g,2t+8) q(g+8,2t+8) q(g,2t+1) q(g+8,2t+1)
//     q(g,2t+9) q(g+8,2t+9), so shifting by 0/4/8/12 and masking 0x000F000F gives the four A registers.
//     Bytes 512..639: for g = 0..7, 16 B of (d, m) fp16 pairs for columns g, g+8 of the tile's two
//     32-input blocks.
//   bf16 (2048 B): k-step s at 512*s, lane L's 16 B = its four A registers.
// Q4_1 product per 32-block b: y += d_b * sum_k x_k q_k + m_b * sum_k x_k, with q entering the
// tensor core exactly (integers 0..15 are exact in bf16) and the per-block scale applied in fp32.
//
// Split K: the K chunks are cut into S equal ranges (S depends on K and N only); each warp computes
// two tiles over one range; the last warp to finish a column pair (arrival counter) adds the S
// partial sums in the fixed order 0..S-1 and applies the epilogue. So a row's result never depends on
// how many rows the pass carries: a batched pass equals single-row passes bit for bit.
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

// ---------------------------------------------------------------------------------------------------
// shared pieces of the product kernels
// ---------------------------------------------------------------------------------------------------

// Activations enter the tensor cores as bf16 B fragments. An fp32 activation x is split into
// hi = bf16(x) and lo = bf16(x - hi) (x - hi is exact in fp32), so hi + lo = x to 2^-17 relative and
// the product runs as two MMAs into the same accumulator. bf16 activations (XIN = 0) take one MMA.
//
// Staged layout, per chunk cc, token tile tt, k-step ks and lane L (token 8tt + L/4, t = L%4):
//   XIN 0: 8 bytes  {x[k0+2t], x[k0+2t+1]}, {x[k0+2t+8], x[k0+2t+9]}
//   XIN 1: 16 bytes {hi pair, hi pair+8, lo pair, lo pair+8}
// at index ((cc*MT + tt)*4 + ks)*32 + L, so a warp reads one k-step's fragments in one conflict-free
// shared load.
__device__ __forceinline__ uint32_t pack_bf16x2(uint16_t lo, uint16_t hi) { return uint32_t(lo) | (uint32_t(hi) << 16); }

// Copy the raw activation slice rows [0, M) x inputs [64*c0, 64*(c0+nch)) into shared memory with
// 16-byte asynchronous copies (one round trip), zero beyond K.
template <int XIN>
__device__ __forceinline__ void stage_raw(uint8_t *raw, const GemmArgs &a, int row0, int c0, int nch) {
    constexpr int E = XIN ? 4 : 2;                     // bytes per element
    const int rowbytes = nch * 64 * E;
    const int k0 = 64 * c0;
    const int kend = min(a.K, 64 * (c0 + nch));
    const int live = (kend - k0) * E;                  // bytes of a row inside K (multiple of 64)
    const int per_row = rowbytes / 16;
    for (int e = threadIdx.x; e < a.M * per_row; e += blockDim.x) {
        const int m = e / per_row, off = (e % per_row) * 16;
        uint8_t *dst = raw + m * rowbytes + off;
        if (off < live)
            cp_async16(dst, reinterpret_cast<const uint8_t *>(a.x) + ((long)(row0 + m) * a.ldx + k0) * E + off);
        else
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_wait_all();
}

template <int XIN>
__device__ __forceinline__ float raw_at(const uint8_t *raw, int rowbytes, int m, int k) {
    if (XIN) return reinterpret_cast<const float *>(raw + m * rowbytes)[k];
    return bf16_to_f32(reinterpret_cast<const uint16_t *>(raw + m * rowbytes)[k]);
}

// Fragments and per-32-block sums from the raw slice (after a barrier).
template <int MT, int XIN>
__device__ __forceinline__ void stage_frags(uint32_t *xs, float *sums, const uint8_t *raw, const GemmArgs &a, int nch,
                                            bool want_sums) {
    constexpr int W = XIN ? 4 : 2;
    const int rowbytes = nch * 64 * (XIN ? 4 : 2);
    for (int e = threadIdx.x; e < nch * MT * 4 * 32; e += blockDim.x) {
        const int L = e & 31, ks = (e >> 5) & 3, tt = (e >> 7) % MT, cc = (e >> 7) / MT;
        const int tok = 8 * tt + (L >> 2), tq = L & 3;
        const int k = 64 * cc + 16 * ks + 2 * tq;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (tok < a.M) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float v0 = raw_at<XIN>(raw, rowbytes, tok, k + 8 * hh);
                const float v1 = raw_at<XIN>(raw, rowbytes, tok, k + 8 * hh + 1);
                const uint16_t h0 = f32_to_bf16(v0), h1 = f32_to_bf16(v1);
                w[hh] = pack_bf16x2(h0, h1);
                if (XIN) w[2 + hh] = pack_bf16x2(f32_to_bf16(v0 - bf16_to_f32(h0)), f32_to_bf16(v1 - bf16_to_f32(h1)));
            }
        }
        uint32_t *d = xs + (size_t)e * W;
        if (XIN) *reinterpret_cast<uint4 *>(d) = make_uint4(w[0], w[1], w[2], w[3]);
        else *reinterpret_cast<uint2 *>(d) = make_uint2(w[0], w[1]);
    }
    if (!want_sums) return;
    for (int e = threadIdx.x; e < nch * 32; e += blockDim.x) {
        const int tok = e & 15, blk = (e >> 4) & 1, cc = e >> 5;
        float s = 0.f;
        if (tok < a.M)
            for (int i = 0; i < 32; ++i) s += raw_at<XIN>(raw, rowbytes, tok, 64 * cc + 32 * blk + i);
        sums[e] = s;
    }
}

// fragment of k-step ks, token tile tt for this lane
template <int XIN>
__device__ __forceinline__ uint4 frag(const uint32_t *xs, int cc, int tt, int ks, int lane, int MT) {
    const size_t e = ((size_t)(cc * MT + tt) * 4 + ks) * 32 + lane;
    if (XIN) return *reinterpret_cast<const uint4 *>(xs + e * 4);
    const uint2 v = *reinterpret_cast<const uint2 *>(xs + e * 2);
    return make_uint4(v.x, v.y, 0u, 0u);
}

template <int XIN>
__device__ __forceinline__ void mma_x(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, const uint4 &b) {
    mma_bf16(d, a0, a1, a2, a3, b.x, b.y);
    if (XIN) mma_bf16(d, a0, a1, a2, a3, b.z, b.w);
}

template <int MT, int XIN>
__device__ __forceinline__ void q41_chunk(float (&acc)[2][MT][4], const uint4 (&nb)[2], const uint4 (&sc)[2],
                                          const uint32_t *xs, const float *sums, int cc, int lane) {
    const int t = lane & 3;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        float2 S[MT];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
            S[tt] = *reinterpret_cast<const float2 *>(sums + (cc * 2 + blk) * 16 + 8 * tt + 2 * t);
        float cb[2][MT][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) cb[j][tt][0] = cb[j][tt][1] = cb[j][tt][2] = cb[j][tt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int ks = 2 * blk + kk;
            uint4 b[MT];
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) b[tt] = frag<XIN>(xs, cc, tt, ks, lane, MT);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t w = ks == 0 ? nb[j].x : ks == 1 ? nb[j].y : ks == 2 ? nb[j].z : nb[j].w;
                const uint32_t a0 = nib_pair_bf16(w), a1 = nib_pair_bf16(w >> 4);
                const uint32_t a2 = nib_pair_bf16(w >> 8), a3 = nib_pair_bf16(w >> 12);
#pragma unroll
                for (int tt = 0; tt < MT; ++tt) mma_x<XIN>(cb[j][tt], a0, a1, a2, a3, b[tt]);
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t dlo = blk ? sc[j].z : sc[j].x, dhi = blk ? sc[j].w : sc[j].y;
            const float2 flo = __half22float2(*reinterpret_cast<__half2 *>(&dlo));   // (d, m) of column g
            const float2 fhi = __half22float2(*reinterpret_cast<__half2 *>(&dhi));   // column g + 8
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
                acc[j][tt][0] = fmaf(flo.y, S[tt].x, fmaf(flo.x, cb[j][tt][0], acc[j][tt][0]));
                acc[j][tt][1] = fmaf(flo.y, S[tt].y, fmaf(flo.x, cb[j][tt][1], acc[j][tt][1]));
                acc[j][tt][2] = fmaf(fhi.y, S[tt].x, fmaf(fhi.x, cb[j][tt][2], acc[j][tt][2]));
                acc[j][tt][3] = fmaf(fhi.y, S[tt].y, fmaf(fhi.x, cb[j][tt][3], acc[j][tt][3]));
            }
        }
    }
}

template <int MT, int XIN>
__device__ __forceinline__ void bf16_chunk(float (&acc)[2][MT][4], const uint4 (&w)[2][4], const uint32_t *xs, int cc,
                                           int lane) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint4 b[MT];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) b[tt] = frag<XIN>(xs, cc, tt, ks, lane, MT);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) mma_x<XIN>(acc[j][tt], w[j][ks].x, w[j][ks].y, w[j][ks].z, w[j][ks].w, b[tt]);
    }
}

// ---------------------------------------------------------------------------------------------------
// split-K product with fused epilogue
// ---------------------------------------------------------------------------------------------------
template <int MT, int EPI>
__device__ __forceinline__ void epilogue(const GemmArgs &a, float (&acc)[2][MT][4], int nt0, int nt1, int ng, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = 8 * tt + 2 * t + (i & 1);
            if (tok >= a.M) continue;
            const int r = g + 8 * (i >> 1);
            if (EPI == EPI_F32) {
                float *y = reinterpret_cast<float *>(a.y) + (long)tok * a.ldy;
                y[16 * nt0 + r] = acc[0][tt][i];
                y[16 * nt1 + r] = acc[1][tt][i];
            } else if (EPI == EPI_GLU) {
                float *y = reinterpret_cast<float *>(a.y) + (long)tok * a.ldy;
                y[16 * ng + r] = silu_f(acc[0][tt][i]) * acc[1][tt][i];
            } else if (EPI == EPI_SILU_MUL) {
                float *y = reinterpret_cast<float *>(a.y) + (long)tok * a.ldy;
                const uint16_t *e = a.ext + (long)tok * a.lde;
                const int n0 = 16 * nt0 + r, n1 = 16 * nt1 + r;
                y[n0] = silu_f(acc[0][tt][i]) * bf16_to_f32(e[n0]);
                y[n1] = silu_f(acc[1][tt][i]) * bf16_to_f32(e[n1]);
            }
        }
}

template <int FMT, int MT, int EPI, int XIN>
__global__ void __launch_bounds__(128) k_gemm(GemmArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2;
    const int s = blockIdx.y;
    const int c0 = int((long)s * a.C / a.S), c1 = int((long)(s + 1) * a.C / a.S);
    const int nch = c1 - c0;
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem);
    float *sums = reinterpret_cast<float *>(smem + (size_t)nch * MT * 4 * 32 * (XIN ? 16 : 8));
    uint8_t *raw = reinterpret_cast<uint8_t *>(sums + nch * 32);

    const int ngroups = a.N / 32;
    const int ng = blockIdx.x * kWarpsPerCta + warp;
    const bool active = ng < ngroups;
    const int nt0 = active ? ((EPI == EPI_GLU) ? ng : 2 * ng) : 0;
    const int nt1 = active ? ((EPI == EPI_GLU) ? ng + ngroups : 2 * ng + 1) : 0;

    // the first weight chunks are requested before the activations are staged, so the two latencies overlap
    constexpr int PQ = 4, PB = 2;
    constexpr int TB = FMT == W_Q41 ? 640 : 2048;
    const uint8_t *base0 = a.img + ((size_t)nt0 * a.C + c0) * TB;
    const uint8_t *base1 = a.img + ((size_t)nt1 * a.C + c0) * TB;
    uint4 nb[PQ][2], sc[PQ][2];
    uint4 w[PB][2][4];
    if (active) {
        if (FMT == W_Q41) {
#pragma unroll
            for (int p = 0; p < PQ; ++p)
                if (p < nch) {
                    nb[p][0] = ldg_stream(base0 + p * 640 + 16 * lane);
                    nb[p][1] = ldg_stream(base1 + p * 640 + 16 * lane);
                    sc[p][0] = ldg_stream(base0 + p * 640 + 512 + 16 * g);
                    sc[p][1] = ldg_stream(base1 + p * 640 + 512 + 16 * g);
                }
        } else {
#pragma unroll
            for (int p = 0; p < PB; ++p)
                if (p < nch)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        w[p][0][ks] = ldg_stream(base0 + p * 2048 + 512 * ks + 16 * lane);
                        w[p][1][ks] = ldg_stream(base1 + p * 2048 + 512 * ks + 16 * lane);
                    }
        }
    }
    pdl_wait();          // the activations are written by the previous kernel
    pdl_trigger();
    stage_raw<XIN>(raw, a, a.x_row0, c0, nch);
    __syncthreads();
    stage_frags<MT, XIN>(xs, sums, raw, a, nch, FMT == W_Q41);
    __syncthreads();
    if (!active) return;

    float acc[2][MT][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) acc[j][tt][0] = acc[j][tt][1] = acc[j][tt][2] = acc[j][tt][3] = 0.f;

    if (FMT == W_Q41) {
        for (int cb = 0; cb < nch; cb += PQ) {
#pragma unroll
            for (int p = 0; p < PQ; ++p) {
                const int cc = cb + p;
                if (cc < nch) {
                    q41_chunk<MT, XIN>(acc, nb[p], sc[p], xs, sums, cc, lane);
                    const int nx = cc + PQ;
                    if (nx < nch) {
                        nb[p][0] = ldg_stream(base0 + (size_t)nx * 640 + 16 * lane);
                        nb[p][1] = ldg_stream(base1 + (size_t)nx * 640 + 16 * lane);
                        sc[p][0] = ldg_stream(base0 + (size_t)nx * 640 + 512 + 16 * g);
                        sc[p][1] = ldg_stream(base1 + (size_t)nx * 640 + 512 + 16 * g);
                    }
                }
            }
        }
    } else {
        for (int cb = 0; cb < nch; cb += PB) {
#pragma unroll
            for (int p = 0; p < PB; ++p) {
                const int cc = cb + p;
                if (cc < nch) {
                    bf16_chunk<MT, XIN>(acc, w[p], xs, cc, lane);
                    const int nx = cc + PB;
                    if (nx < nch)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            w[p][0][ks] = ldg_stream(base0 + (size_t)nx * 2048 + 512 * ks + 16 * lane);
                            w[p][1][ks] = ldg_stream(base1 + (size_t)nx * 2048 + 512 * ks + 16 * lane);
                        }
                }
            }
        }
    }

    if (a.S > 1) {
        const int t = lane & 3;
        float *P0 = a.part + (size_t)s * a.M * a.N;
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = 8 * tt + 2 * t + (i & 1);
                if (tok >= a.M) continue;
                const int r = g + 8 * (i >> 1);
                P0[(long)tok * a.N + 16 * nt0 + r] = acc[0][tt][i];
                P0[(long)tok * a.N + 16 * nt1 + r] = acc[1][tt][i];
            }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = (atomicAdd(a.cnt + ng, 1) == a.S - 1);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) return;
        __threadfence();
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = 8 * tt + 2 * t + (i & 1);
                if (tok >= a.M) continue;
                const int r = g + 8 * (i >> 1);
                float v0 = 0.f, v1 = 0.f;
                const float *Pb = a.part + (long)tok * a.N;
                const size_t stride = (size_t)a.M * a.N;
                int s2 = 0;
                for (; s2 + 8 <= a.S; s2 += 8) {
                    float u0[8], u1[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        u0[q] = __ldcg(Pb + (s2 + q) * stride + 16 * nt0 + r);
                        u1[q] = __ldcg(Pb + (s2 + q) * stride + 16 * nt1 + r);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) v0 += u0[q], v1 += u1[q];
                }
                for (; s2 < a.S; ++s2) {
                    v0 += __ldcg(Pb + s2 * stride + 16 * nt0 + r);
                    v1 += __ldcg(Pb + s2 * stride + 16 * nt1 + r);
                }
                acc[0][tt][i] = v0;
                acc[1][tt][i] = v1;
            }
        if (lane == 0) a.cnt[ng] = 0;
    }
    epilogue<MT, EPI>(a, acc, nt0, nt1, ng, lane);
}

// ---------------------------------------------------------------------------------------------------
// bf16 head: logits of M rows over the vocabulary, fused with the first-maximum argmax and, for a
// verify, the longest-prefix acceptance.
// ---------------------------------------------------------------------------------------------------
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

template <int MT>
__device__ __forceinline__ void stage_head_x(uint32_t *xs, const GemmArgs &a) {
    for (int e = threadIdx.x; e < a.C * MT * 4 * 32; e += blockDim.x) {
        const int L = e & 31, ks = (e >> 5) & 3, tt = (e >> 7) % MT, cc = (e >> 7) / MT;
        const int tok = 8 * tt + (L >> 2), tq = L & 3;
        const int k = 64 * cc + 16 * ks + 2 * tq;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (tok < a.M) {
            const float *xr = reinterpret_cast<const float *>(a.x) + (long)(a.x_row0 + tok) * a.ldx;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int kk = k + 8 * hh;
                const float2 v = kk < a.K ? *reinterpret_cast<const float2 *>(xr + kk) : make_float2(0.f, 0.f);
                const uint16_t h0 = f32_to_bf16(v.x), h1 = f32_to_bf16(v.y);
                w[hh] = pack_bf16x2(h0, h1);
                w[2 + hh] = pack_bf16x2(f32_to_bf16(v.x - bf16_to_f32(h0)), f32_to_bf16(v.y - bf16_to_f32(h1)));
            }
        }
        *reinterpret_cast<uint4 *>(xs + (size_t)e * 4) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int MT>
__global__ void __launch_bounds__(128) k_head(GemmArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float wval[kWarpsPerCta][kMaxRows];
    __shared__ int widx[kWarpsPerCta][kMaxRows];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem);

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
    // the activations are staged while the first weight chunks are in flight
    pdl_wait();
    pdl_trigger();
    stage_head_x<MT>(xs, a);
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
                bf16_chunk<MT, 1>(acc, w[p], xs, c, lane);
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
int gemm_splits(int C, int N, int fmt) {
    (void)fmt;
    const int ngroups = N / 32;
    int S = (kSplitTargetWarps + ngroups - 1) / ngroups;
    const int smin = (C + kMaxChunksPerSplit - 1) / kMaxChunksPerSplit;   // bound shared memory
    const int smax = C / 4 > 0 ? C / 4 : 1;                                // at least 4 chunks a warp
    if (S > smax) S = smax;
    if (S < smin) S = smin;
    if (S < 1) S = 1;
    if (S > C) S = C;
    return S;
}

size_t gemm_scratch_floats(int S, int M, int N) { return S > 1 ? (size_t)S * M * N : 0; }

size_t gemm_smem(int C, int S, int MT, int XIN, int fmt, int M) {
    (void)fmt;
    const int maxch = (C + S - 1) / S;
    return (size_t)maxch * MT * 4 * 32 * (XIN ? 16 : 8) + (size_t)maxch * 128 + (size_t)M * maxch * 64 * (XIN ? 4 : 2);
}

template <int FMT, int MT, int EPI, int XIN>
static cudaError_t run_gemm(const GemmArgs &a, cudaStream_t s) {
    const size_t smem = gemm_smem(a.C, a.S, MT, XIN, FMT, a.M);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm<FMT, MT, EPI, XIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int ngroups = a.N / 32;
    dim3 grid((ngroups + kWarpsPerCta - 1) / kWarpsPerCta, a.S);
    return launch_pdl(k_gemm<FMT, MT, EPI, XIN>, grid, dim3(128), smem, s, a);
}

template <int MT>
static cudaError_t run_head(const GemmArgs &a, cudaStream_t s) {
    const size_t smem = (size_t)a.C * MT * 2048;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_head<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int per_sm = smem <= 48 * 1024 ? 4 : (smem <= 100 * 1024 ? 2 : 1);
    int grid = 152 * per_sm;
    const int ntiles = a.N / 16;
    if (grid * kWarpsPerCta > ntiles) grid = (ntiles + kWarpsPerCta - 1) / kWarpsPerCta;
    return launch_pdl(k_head<MT>, dim3(grid), dim3(128), smem, s, a);
}

int head_grid(int C, int M, int N) {
    const int MT = M > 8 ? 2 : 1;
    const size_t smem = (size_t)C * MT * 2048;
    const int per_sm = smem <= 48 * 1024 ? 4 : (smem <= 100 * 1024 ? 2 : 1);
    int grid = 152 * per_sm;
    const int ntiles = N / 16;
    if (grid * kWarpsPerCta > ntiles) grid = (ntiles + kWarpsPerCta - 1) / kWarpsPerCta;
    return grid;
}

cudaError_t launch_gemm(int fmt, int epi, int xin, const GemmArgs &a, cudaStream_t s) {
    const bool two = a.M > 8;
    if (epi == EPI_ARGMAX) return two ? run_head<2>(a, s) : run_head<1>(a, s);
#define DFL_GEMM_CASE(F, E, X)                                                      \
    if (fmt == F && epi == E && xin == X) return two ? run_gemm<F, 2, E, X>(a, s) : run_gemm<F, 1, E, X>(a, s);
    DFL_GEMM_CASE(W_Q41, EPI_F32, 1)
    DFL_GEMM_CASE(W_Q41, EPI_GLU, 1)
    DFL_GEMM_CASE(W_Q41, EPI_SILU_MUL, 1)
    DFL_GEMM_CASE(W_BF16, EPI_F32, 1)
    DFL_GEMM_CASE(W_Q41, EPI_F32, 0)
#undef DFL_GEMM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace dfl
