// rows.cu -- row-wise pieces of the step: embedding and per-layer-embedding gather, the residual /
// RMSNorm / layer-scalar / tap row kernel, query-key norm + rotary embedding + KV append, split-KV
// grouped-query attention over per-layer planes, temperature sampling with prefix acceptance.
//
// Sources (pages, by title and section): 1bit engine PR "npu forward: Gemma4 verifies a draft in one
// batched pass; KV row width per layer" ("What changes": per-layer inputs built per row, PLE gate and
// projection then the layer scalar, KV-shared layers read the owner's cache and append nothing, per
// layer KV width; reviewer excerpt: sandwich norms on Gemma4 layers); model card
// "Nemotron-3.5-Bolt-E4B-DFlash-NPU2" (draft: Qwen3-style layers, window 1024, block of 8; "How it is
// used": every position sampled and compared with the draft when a sampler is on).
#include "common.cuh"

namespace dfl {

// ---------------------------------------------------------------------------------------------------
__global__ void k_set_state(DevState *st, SetStateArgs a) {
    pdl_wait();
    pdl_trigger();
    const int i = threadIdx.x;
    int r = 0;
    if (i < kMaxRows) r = a.use_draft_rows ? (i == 0 ? st->last_tok : st->props[i - 1]) : a.rows[i];
    __syncwarp();
    if (i < kMaxRows) st->rows[i] = r;
    if (i == 0) {
        st->n = a.n;
        st->k = a.k;
        st->draft_n = a.draft_n;
        st->ctx_rows = a.ctx_rows;
        st->sampled = a.sampled;
        st->temperature = a.temperature;
        st->seed = a.seed;
        if (a.last_tok >= 0) st->last_tok = a.last_tok;
    }
}

cudaError_t launch_set_state(DevState *st, const SetStateArgs &a, cudaStream_t s) {
    return launch_pdl(k_set_state, dim3(1), dim3(32), 0, s, st, a);
}

// planted drafts: the proposals for positions n+1..n+count become table[n+1..n+count]
__global__ void k_plant(DevState *st, const int32_t *table, int count) {
    pdl_wait();
    pdl_trigger();
    const int i = threadIdx.x;
    if (i < count) st->props[i] = table[st->n + 1 + i];
}

cudaError_t launch_plant(DevState *st, const int32_t *table, int count, cudaStream_t s) {
    return launch_pdl(k_plant, dim3(1), dim3(32), 0, s, st, table, count);
}

// ---------------------------------------------------------------------------------------------------
// x[m] = emb[token_m] * scale (fp32); the row's per-layer-embedding inputs are a plain table row.
__global__ void k_embed(EmbedArgs a) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x;
    const int tok = a.use_draft ? (m == 0 ? a.st->last_tok : a.mask_token) : a.st->rows[m];
    const uint16_t *e = a.emb + (long)tok * a.H;
    for (int h = threadIdx.x; h < a.H; h += blockDim.x) a.x[(long)m * a.H + h] = bf16_to_f32(e[h]) * a.scale;
    if (a.ple) {
        const uint16_t *p = a.ple + (long)tok * a.ple_w;
        for (int h = threadIdx.x; h < a.ple_w; h += blockDim.x) a.ple_out[(long)m * a.ple_w + h] = p[h];
    }
}

cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t s) {
    return launch_pdl(k_embed, dim3(a.M), dim3(256), 0, s, a);
}

// ---------------------------------------------------------------------------------------------------
// Residual row kernel:
//   x += RMSNorm(y, w_post) (or x += y), x *= lambda, tap = bf16(x), out = bf16(RMSNorm(x, w_next)).
constexpr int kRowThreads = 256;
constexpr int kRowMaxPer = 16;   // hidden <= 4096

__global__ void __launch_bounds__(kRowThreads) k_rows(RowArgs a) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[33];
    const int m = blockIdx.x;
    const bool live = !a.rows_from_ctx || m < a.st->ctx_rows;
    const int per = (a.H + kRowThreads - 1) / kRowThreads;
    float xv[kRowMaxPer];
    float *x = a.x ? a.x + (long)m * a.H : nullptr;
#pragma unroll
    for (int i = 0; i < kRowMaxPer; ++i) {
        const int h = threadIdx.x + i * kRowThreads;
        xv[i] = (i < per && h < a.H && x) ? x[h] : 0.f;
    }
    if (a.y) {
        const float *y = a.y + (long)m * a.ldy;
        float yv[kRowMaxPer];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < kRowMaxPer; ++i) {
            const int h = threadIdx.x + i * kRowThreads;
            yv[i] = (i < per && h < a.H) ? y[h] : 0.f;
            ss += yv[i] * yv[i];
        }
        float r = 1.f;
        if (a.w_post) r = 1.0f / sqrtf(block_sum(ss, red) / a.H + a.eps);
#pragma unroll
        for (int i = 0; i < kRowMaxPer; ++i) {
            const int h = threadIdx.x + i * kRowThreads;
            if (i < per && h < a.H) xv[i] = a.w_post ? xv[i] + (yv[i] * r) * bf16_to_f32(a.w_post[h]) : xv[i] + yv[i];
        }
    }
    if (a.lambda != 1.0f) {
#pragma unroll
        for (int i = 0; i < kRowMaxPer; ++i) xv[i] *= a.lambda;
    }
    if (x && (a.y || a.lambda != 1.0f)) {
#pragma unroll
        for (int i = 0; i < kRowMaxPer; ++i) {
            const int h = threadIdx.x + i * kRowThreads;
            if (i < per && h < a.H) x[h] = xv[i];
        }
    }
    if (a.tap && live) {
        const int pos = (a.pos_from_ctx ? a.st->draft_n : a.st->n) + m;
        float *tp = a.tap + (long)pos * a.ld_tap + a.tap_off;
#pragma unroll
        for (int i = 0; i < kRowMaxPer; ++i) {
            const int h = threadIdx.x + i * kRowThreads;
            if (i < per && h < a.H) tp[h] = xv[i];
        }
    }
    if (a.outf) {
        float r = 1.f;
        if (a.w_next) {
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < kRowMaxPer; ++i) ss += xv[i] * xv[i];
            r = 1.0f / sqrtf(block_sum(ss, red) / a.H + a.eps);
        }
        const int row = a.out_row0 + m;
#pragma unroll
        for (int i = 0; i < kRowMaxPer; ++i) {
            if (i >= per) break;
            const int h = threadIdx.x + i * kRowThreads;
            float v = 0.f;
            if (h < a.H && live) v = a.w_next ? (xv[i] * r) * bf16_to_f32(a.w_next[h]) : xv[i];
            if (h < a.H) act_store(a.outf, a.H, row, h, v);
            const float sg = half_warp_sum(v);
            if (h < a.H && (h & 15) == 0) a.outs[(h >> 4) * kMaxRows + row] = sg;
        }
    }
}

cudaError_t launch_rows(const RowArgs &a, cudaStream_t s) {
    if (a.H > kRowThreads * kRowMaxPer || a.H % 16) return cudaErrorInvalidValue;
    return launch_pdl(k_rows, dim3(a.M), dim3(kRowThreads), 0, s, a);
}

// dst row (row0 + m) = RMSNorm(src[m], w) for live rows (m < st->ctx_rows when live_from_ctx), zeros
// otherwise, in operand format.
__global__ void __launch_bounds__(kRowThreads) k_cast_rows(const float *src, int ld_src, int H, const uint16_t *w,
                                                           float eps, uint32_t *dstf, float *dsts, int row0,
                                                           const DevState *st, int live_from_ctx) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[33];
    const int m = blockIdx.x;
    const bool live = !live_from_ctx || m < st->ctx_rows;
    const int per = (H + kRowThreads - 1) / kRowThreads;
    float v[kRowMaxPer];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kRowMaxPer; ++i) {
        const int h = threadIdx.x + i * kRowThreads;
        v[i] = (i < per && h < H) ? src[(long)m * ld_src + h] : 0.f;
        ss += v[i] * v[i];
    }
    const float r = 1.0f / sqrtf(block_sum(ss, red) / H + eps);
#pragma unroll
    for (int i = 0; i < kRowMaxPer; ++i) {
        if (i >= per) break;
        const int h = threadIdx.x + i * kRowThreads;
        const float o = (h < H && live) ? (v[i] * r) * bf16_to_f32(w[h]) : 0.f;
        if (h < H) act_store(dstf, H, row0 + m, h, o);
        const float sg = half_warp_sum(o);
        if (h < H && (h & 15) == 0) dsts[(h >> 4) * kMaxRows + row0 + m] = sg;
    }
}

cudaError_t launch_cast_rows(const float *src, int ld_src, int M, int H, const uint16_t *w_norm, float eps,
                             uint32_t *dstf, float *dsts, int row0, const DevState *st, int live_from_ctx,
                             cudaStream_t s) {
    if (H > kRowThreads * kRowMaxPer || H % 16) return cudaErrorInvalidValue;
    return launch_pdl(k_cast_rows, dim3(M), dim3(kRowThreads), 0, s, src, ld_src, H, w_norm, eps, dstf, dsts, row0, st,
                      live_from_ctx);
}

// ---------------------------------------------------------------------------------------------------
// Per head: RMSNorm over the head dimension, then the half-split rotary embedding at the row's
// absolute position, from a (cos, sin) table computed in double precision. Keys and values are
// stored into their plane slot (pos % cap), or into the block store (slot = row).
__global__ void k_qk(QkArgs a) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[33];
    const int m = blockIdx.x, h = blockIdx.y, i = threadIdx.x, half = a.hd / 2;
    const bool live = !a.live_from_ctx || m < a.st->ctx_rows;
    if (!live) return;
    const int pos = (a.pos_mode == 2 ? a.st->draft_n : a.st->n) + m;
    const float *row = a.qkv + (long)(a.row0 + m) * a.ldq;
    const int nqh = a.q_out ? a.nq : 0;
    const bool is_q = h < nqh;
    const int hk = h - nqh;
    const float *src = is_q ? row + h * a.hd : row + (a.nq + hk) * a.hd;
    const uint16_t *w = is_q ? a.q_norm : a.k_norm;
    float u0 = src[i], u1 = src[i + half];
    const float r = 1.0f / sqrtf(block_sum(u0 * u0 + u1 * u1, red) / a.hd + a.eps);
    u0 = (u0 * r) * bf16_to_f32(w[i]);
    u1 = (u1 * r) * bf16_to_f32(w[i + half]);
    const float2 cs = a.rope[(long)pos * half + i];
    const float o0 = u0 * cs.x - u1 * cs.y, o1 = u0 * cs.y + u1 * cs.x;
    if (is_q) {
        float *q = a.q_out + ((long)m * a.nq + h) * a.hd;
        q[i] = o0;
        q[i + half] = o1;
    } else {
        const long slot = a.cap > 0 ? (long)(pos % a.cap) : (long)m;
        float *k = a.k_store + (slot * a.nkv + hk) * a.hd;
        float *v = a.v_store + (slot * a.nkv + hk) * a.hd;
        const float *vs = row + (a.nq + a.nkv + hk) * a.hd;
        k[i] = o0;
        k[i + half] = o1;
        v[i] = vs[i];
        v[i + half] = vs[i + half];
    }
}

cudaError_t launch_qk(const QkArgs &a, cudaStream_t s) {
    const int heads = (a.q_out ? a.nq : 0) + (a.k_store ? a.nkv : 0);
    if (heads == 0) return cudaSuccess;
    if (a.hd / 2 < 32 || a.hd / 2 > 1024 || (a.hd / 2) % 32) return cudaErrorInvalidValue;
    return launch_pdl(k_qk, dim3(a.M, heads), dim3(a.hd / 2), 0, s, a);
}

// ---------------------------------------------------------------------------------------------------
// Attention. Work item = (query head, chunk of kAttnChunk keys). The chunks cover, for the target
// (mode 0), positions lo..n+M-1 of the head's plane with lo = max(0, n-window+1) on sliding layers, each
// row m at position n+m seeing keys max(0, n+m-window+1)..n+m (all of 0..n+m on full layers); for the
// draft (mode 1), context positions max(0, n-window)..n-1 for every row plus one chunk of the block's
// own keys, all visible. Each item writes its softmax partial (max, sum, sum of p*v); the last item of
// a head (arrival counter) combines the chunks in chunk order and writes bf16 outputs.
constexpr int kAttnThreads = 128;

__device__ __forceinline__ void attn_range(const AttnArgs &a, int n, int &lo, int &nA, int &nchunks) {
    if (a.mode == 0) {
        lo = a.window > 0 ? max(0, n - a.window + 1) : 0;
        nA = n + a.M - lo;
        nchunks = (nA + kAttnChunk - 1) / kAttnChunk;
    } else {
        lo = a.window > 0 ? max(0, n - a.window) : 0;
        nA = n - lo;
        nchunks = (nA + kAttnChunk - 1) / kAttnChunk + 1;
    }
}

__global__ void __launch_bounds__(kAttnThreads) k_attn(AttnArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_last;
    const int hd = a.hd, ks = hd + 1;   // key row stride in floats (odd: conflict-free column reads)
    float *Ks = reinterpret_cast<float *>(smem);
    float *Vs = Ks + kAttnChunk * ks;
    float *qs = Vs + kAttnChunk * ks;     // [M][hd]
    float *ps = qs + a.M * hd;            // [M][kAttnChunk]
    const int n = a.st->n;
    int lo, nA, nchunks;
    attn_range(a, n, lo, nA, nchunks);
    const int grp = a.nq / a.nkv;
    const int items = a.nq * nchunks;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kAttnThreads / 32;

    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int h = it / nchunks, c = it % nchunks, g = h / grp;
        const bool blockchunk = (a.mode == 1 && c == nchunks - 1);
        const int j0 = blockchunk ? 0 : lo + c * kAttnChunk;
        const int nk = blockchunk ? a.nB : min(kAttnChunk, lo + nA - j0);
        __syncthreads();
        // keys and values of the chunk, and the queries of this head
        for (int e = tid; e < nk * hd; e += kAttnThreads) {
            const int jj = e / hd, d = e % hd;
            long off;
            const float *kb, *vb;
            if (blockchunk) {
                off = ((long)jj * a.nkv + g) * hd;
                kb = a.kB;
                vb = a.vB;
            } else {
                const long slot = (j0 + jj) % a.capA;
                off = (slot * a.nkv + g) * hd;
                kb = a.kA;
                vb = a.vA;
            }
            Ks[jj * ks + d] = kb[off + d];
            Vs[jj * ks + d] = vb[off + d];
        }
        for (int e = tid; e < a.M * hd; e += kAttnThreads) {
            const int m = e / hd, d = e % hd;
            qs[e] = a.q[((long)m * a.nq + h) * hd + d];
        }
        __syncthreads();
        // scores: thread -> key jj = lane, rows warp, warp + NW, ...
        {
            const int jj = lane;
            float sc[kMaxRows / NW];
#pragma unroll
            for (int r = 0; r < kMaxRows / NW; ++r) sc[r] = 0.f;
            if (jj < nk) {
                for (int d = 0; d < hd; ++d) {
                    const float kv = Ks[jj * ks + d];
#pragma unroll
                    for (int r = 0; r < kMaxRows / NW; ++r) {
                        const int m = warp + r * NW;
                        if (m < a.M) sc[r] = fmaf(qs[m * hd + d], kv, sc[r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kMaxRows / NW; ++r) {
                const int m = warp + r * NW;
                if (m >= a.M) continue;
                bool vis = jj < nk;
                if (vis && a.mode == 0) {
                    const int j = j0 + jj, p = n + m;
                    vis = j <= p && (a.window <= 0 || j > p - a.window);
                }
                ps[m * kAttnChunk + jj] = vis ? sc[r] * a.scale : -INFINITY;
            }
        }
        __syncthreads();
        // softmax partial per row: warp w takes rows w, w + NW, ...
        float *pml = a.part_ml + ((long)h * a.max_chunks + c) * a.M * 2;
        for (int m = warp; m < a.M; m += NW) {
            const float v = ps[m * kAttnChunk + lane];
            float mx = v;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float p = mx == -INFINITY ? 0.f : expf(v - mx);
            float sm = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
            ps[m * kAttnChunk + lane] = p;
            if (lane == 0) pml[m * 2] = mx, pml[m * 2 + 1] = sm;
        }
        __syncthreads();
        // p . V, keys in ascending order
        float *pacc = a.part_acc + ((long)h * a.max_chunks + c) * a.M * hd;
        for (int e = tid; e < a.M * hd; e += kAttnThreads) {
            const int m = e / hd, d = e % hd;
            float acc = 0.f;
            for (int jj = 0; jj < nk; ++jj) acc = fmaf(ps[m * kAttnChunk + jj], Vs[jj * ks + d], acc);
            pacc[e] = acc;
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = (atomicAdd(a.cnt + h, 1) == nchunks - 1);
        __syncthreads();
        if (s_last) {
            __threadfence();
            for (int e = tid; e < a.M * hd; e += kAttnThreads) {
                const int m = e / hd, d = e % hd;
                float mt = -INFINITY;
                for (int c2 = 0; c2 < nchunks; ++c2)
                    mt = fmaxf(mt, __ldcg(a.part_ml + (((long)h * a.max_chunks + c2) * a.M + m) * 2));
                float num = 0.f, den = 0.f;
                for (int c2 = 0; c2 < nchunks; ++c2) {
                    const long b = ((long)h * a.max_chunks + c2) * a.M + m;
                    const float mc = __ldcg(a.part_ml + b * 2);
                    const float f = mc == -INFINITY ? 0.f : expf(mc - mt);
                    den = fmaf(__ldcg(a.part_ml + b * 2 + 1), f, den);
                    num = fmaf(__ldcg(a.part_acc + b * hd + d), f, num);
                }
                const float o = num / den;
                const int col = h * hd + d;
                act_store(a.outf, a.nq * hd, m, col, o);
                const float sg = half_warp_sum(o);
                if ((col & 15) == 0) a.outs[(col >> 4) * kMaxRows + m] = sg;
            }
            if (tid == 0) a.cnt[h] = 0;
        }
    }
}

size_t attn_smem(int M, int hd) { return ((size_t)2 * kAttnChunk * (hd + 1) + (size_t)M * hd + (size_t)M * kAttnChunk) * 4; }

cudaError_t launch_attn(const AttnArgs &a, int grid, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    if (a.hd % 32 || a.M > kMaxRows || a.nB > kAttnChunk || (a.M * a.hd) % 32) return cudaErrorInvalidValue;
    return launch_pdl(k_attn, dim3(grid), dim3(kAttnThreads), attn_smem(a.M, a.hd), s, a);
}

// ---------------------------------------------------------------------------------------------------
// Sampling. SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) as a counter-based uniform per position.
__device__ __forceinline__ unsigned long long splitmix64(unsigned long long x) {
    unsigned long long z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

constexpr int kSampleThreads = 1024;

// Row m's token for position n+m+1: the smallest j whose running sum of exp((l_j - max)/T) exceeds
// U * total (running sums in double; each thread sums a contiguous segment, then a block scan).
__global__ void __launch_bounds__(kSampleThreads) k_sample(SampleArgs a) {
    pdl_wait();
    pdl_trigger();
    __shared__ float redf[33];
    __shared__ double wsum[32];
    __shared__ int s_tok, s_last;
    const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *l = a.logits + (long)m * a.ld;
    const float T = a.st->temperature;
    // max
    float mx = -INFINITY;
    for (int j = tid; j < a.V; j += kSampleThreads) mx = fmaxf(mx, l[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) redf[warp] = mx;
    __syncthreads();
    if (tid < 32) {
        float v = redf[tid];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (tid == 0) redf[32] = v;
    }
    __syncthreads();
    mx = redf[32];
    const int seg = (a.V + kSampleThreads - 1) / kSampleThreads;
    const int j0 = tid * seg, j1 = min(a.V, j0 + seg);
    double s = 0.0;
    for (int j = j0; j < j1; ++j) s += (double)expf((l[j] - mx) / T);
    // inclusive scan over threads (warp shuffles, then warp totals)
    double inc = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    if (tid == 0) s_tok = -1;
    __syncthreads();
    double before = 0.0, total = 0.0;
    for (int w = 0; w < kSampleThreads / 32; ++w) {
        if (w < warp) before += wsum[w];
        total += wsum[w];
    }
    inc += before;
    const double excl = inc - s;
    const int pos = a.st->n + m + 1;
    const double u = (double)(splitmix64(a.st->seed ^ ((unsigned long long)pos * 0x9E3779B97F4A7C15ull)) >> 11) *
                     (1.0 / 9007199254740992.0);
    const double thr = u * total;
    if (excl <= thr && thr < inc) {
        double c = excl;
        int tok = j1 - 1;
        for (int j = j0; j < j1; ++j) {
            c += (double)expf((l[j] - mx) / T);
            if (c > thr) { tok = j; break; }
        }
        s_tok = tok;
    }
    __syncthreads();
    if (tid == 0) {
        int tok = s_tok;
        if (tok < 0) {   // rounding left u * total at or past the end: the last token with p > 0
            tok = a.V - 1;
            while (tok > 0 && expf((l[tok] - mx) / T) == 0.f) --tok;
        }
        a.st->target[m] = tok;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(a.cnt, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (s_last && tid == 0) {
        __threadfence();
        int acc_len = 0;
        while (acc_len + 1 < a.M && a.st->rows[acc_len + 1] == a.st->target[acc_len]) ++acc_len;
        a.st->accepted = acc_len;
        *a.cnt = 0;
    }
}

cudaError_t launch_sample(const SampleArgs &a, cudaStream_t s) {
    return launch_pdl(k_sample, dim3(a.M), dim3(kSampleThreads), 0, s, a);
}

// ---------------------------------------------------------------------------------------------------
// (cos, sin) of pos * base^(-2i/d) in double precision, stored as float.
__global__ void k_rope_table(float2 *tab, int max_pos, int hd, double base) {
    const long e = blockIdx.x * (long)blockDim.x + threadIdx.x;
    const int half = hd / 2;
    if (e >= (long)max_pos * half) return;
    const int pos = int(e / half), i = int(e % half);
    const double theta = pow(base, -2.0 * i / hd);
    double sn, cs;
    sincos((double)pos * theta, &sn, &cs);
    tab[e] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(float2 *tab, int max_pos, int hd, double base, cudaStream_t s) {
    const long n = (long)max_pos * (hd / 2);
    k_rope_table<<<unsigned((n + 255) / 256), 256, 0, s>>>(tab, max_pos, hd, base);
    return cudaGetLastError();
}

}  // namespace dfl

namespace dfl {

// dst row m = taps row of position st->draft_n + m for m < st->ctx_rows, zeros for the other rows, in
// operand format (the fc product is bf16-weighted: no sums needed).
__global__ void k_copy_taps(const float *taps, int ld, const DevState *st, uint32_t *dstf) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x;
    const bool live = m < st->ctx_rows;
    const float *src = taps + (long)(st->draft_n + (live ? m : 0)) * ld;
    for (int i = threadIdx.x; i < ld; i += blockDim.x) act_store(dstf, ld, m, i, live ? src[i] : 0.f);
}

cudaError_t launch_copy_taps(const float *taps, int ld, const DevState *st, int M, uint32_t *dstf, cudaStream_t s) {
    if (ld % 16) return cudaErrorInvalidValue;
    return launch_pdl(k_copy_taps, dim3(M), dim3(256), 0, s, taps, ld, st, dstf);
}

}  // namespace dfl
