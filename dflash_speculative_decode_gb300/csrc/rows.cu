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
#include "rowstep.cuh"

namespace dfl {

// ---------------------------------------------------------------------------------------------------
__global__ void k_set_state(DevState *st, SetStateArgs a) {
    pdl_trigger();
    pdl_wait();
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
    pdl_trigger();
    pdl_wait();
    const int i = threadIdx.x;
    if (i < count) st->props[i] = table[st->n + 1 + i];
}

cudaError_t launch_plant(DevState *st, const int32_t *table, int count, cudaStream_t s) {
    return launch_pdl(k_plant, dim3(1), dim3(32), 0, s, st, table, count);
}

// ---------------------------------------------------------------------------------------------------
// x[m] = emb[token_m] * scale (fp32); the row's per-layer-embedding inputs are a plain table row.
__global__ void k_embed(EmbedArgs a) {
    pdl_trigger();
    pdl_wait();
    stamp_ready(a.ps);
    const int m = blockIdx.x;
    const int tok = a.use_draft ? (m == 0 ? a.st->last_tok : a.mask_token) : a.tokens ? a.tokens[m] : a.st->rows[m];
    const uint16_t *e = a.emb + (long)tok * a.H;
    for (int h = threadIdx.x; h < a.H; h += blockDim.x) a.x[(long)m * a.H + h] = bf16_to_f32(e[h]) * a.scale;
    if (a.ple) {
        const uint16_t *p = a.ple + (long)tok * a.ple_w;
        for (int h = threadIdx.x; h < a.ple_w; h += blockDim.x) a.ple_out[(long)m * a.ple_w + h] = p[h];
    }
    stamp_done(a.ps);
}

cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t s) {
    return launch_pdl(k_embed, dim3(a.M), dim3(256), 0, s, a);
}

// ---------------------------------------------------------------------------------------------------
// thread-block cluster helpers
// ---------------------------------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// load a float from the shared memory of CTA `rank` of this cluster, at the offset of `p` in ours
__device__ __forceinline__ float ld_cluster(const float *p, unsigned rank) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(p));
    unsigned ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_cluster_pdl(void (*kernel)(KArgs...), dim3 grid, int cluster, int block, size_t smem,
                                      cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = cluster;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------------------------------
// Residual row kernel:
//   x += RMSNorm(y, w_post) (or x += y), x *= lambda, tap = x, out = RMSNorm(x, w_next) in operand format.
// One CTA per row, H/4 threads, each four consecutive columns (128-bit loads and stores). The row sums
// are block sums in a fixed order, so the result does not depend on how many rows the pass carries.
// ---------------------------------------------------------------------------------------------------
constexpr int kRowThreads = 256;   // k_cast_rows
constexpr int kRowMaxPer = 32;     // k_cast_rows: hidden <= 8192

// MAXT bounds the block so that PER slots a thread fit its registers without spilling
template <int PER, int MAXT>
__global__ void __launch_bounds__(MAXT) k_rows(RowArgs a) {
    __shared__ float red[33];
    __shared__ float4 red4[33];
    // the norm weights are immutable: their loads (often from HBM) go out before the dependency wait
    float4 wp[PER], wn[PER];
    row_weights<PER>(a, wp, wn);
    pdl_trigger();
    pdl_wait();
    stamp_ready(a.ps);
    row_step<PER, 8 / PER>(a, blockIdx.x, wp, wn, red, red4);
    stamp_done(a.ps);
}

// One CTA per row: H/4 slots, one per thread up to hidden 4096, two up to 6144 (at most 768 threads),
// three up to 8192 (at most 704 threads).
cudaError_t launch_rows(const RowArgs &a, cudaStream_t s) {
    // rows past 16 only with fp32 output (the operand format holds 16 rows)
    if (a.H % 128 || a.H > 8192 || a.M < 1 || (a.M > kMaxRows && (a.outf || a.out_row0)) || a.M > 65535)
        return cudaErrorInvalidValue;
    if (a.H <= 4096) return launch_pdl(k_rows<1, 1024>, dim3(a.M), dim3(a.H / 4), 0, s, a);
    if (a.H <= 6144) return launch_pdl(k_rows<2, 768>, dim3(a.M), dim3((a.H / 8 + 31) / 32 * 32), 0, s, a);
    return launch_pdl(k_rows<3, 704>, dim3(a.M), dim3((a.H / 12 + 31) / 32 * 32), 0, s, a);
}

// dst row (row0 + m) = RMSNorm(src[m], w) for live rows (m < st->ctx_rows when live_from_ctx), zeros
// otherwise, in operand format.
__global__ void __launch_bounds__(kRowThreads) k_cast_rows(const float *src, int ld_src, int H, const uint16_t *w,
                                                           float eps, uint32_t *dstf, float *dsts, int row0,
                                                           const DevState *st, int live_from_ctx) {
    pdl_trigger();
    pdl_wait();
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
        const float hl = h < H ? act_store(dstf, H, row0 + m, h, o) : 0.f;
        const float sg = half_warp_sum(hl);
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
    __shared__ float red[33];
    const int m = blockIdx.x, h = blockIdx.y, i = threadIdx.x, half = a.hd / 2;
    // Immutable inputs go out before the dependency wait: the norm weights, and the rotation row of the
    // row's position (the position counters were set before the pass began, and every kernel of the pass
    // waits for its predecessor, so they are final here).
    const int nqh0 = a.q_out ? a.nq : 0;
    const uint16_t *w0 = h < nqh0 ? a.q_norm : a.k_norm;
    const float wlo = bf16_to_f32(w0[i]), whi = bf16_to_f32(w0[i + half]);
    const int pos = (a.pos_mode == 2 ? a.st->draft_n : a.st->n) + m;
    const float2 cs = a.rope[(long)pos * half + i];
    pdl_trigger();
    pdl_wait();
    stamp_ready(a.ps);
    const bool live = !a.live_from_ctx || m < a.st->ctx_rows;
    if (!live) {
        stamp_done(a.ps);
        return;
    }
    const int rr = a.row0 + m;
    // column c of this row of the product (plain rows or segment partials); kept for inspection
    auto val = [&](int c) -> float {
        const float v = a.qp.part ? part_sum(a.qp, rr, c) : a.qkv[(long)rr * a.ldq + c];
        if (a.qkv_out) a.qkv_out[(long)rr * a.ldq + c] = v;
        return v;
    };
    const int nqh = a.q_out ? a.nq : 0;
    const bool is_q = h < nqh;
    const int hk = h - nqh;
    const int c0 = is_q ? h * a.hd : (a.nq + hk) * a.hd;
    float u0 = val(c0 + i), u1 = val(c0 + i + half);
    const float r = 1.0f / sqrtf(block_sum(u0 * u0 + u1 * u1, red) / a.hd + a.eps);
    u0 = (u0 * r) * wlo;
    u1 = (u1 * r) * whi;
    const float o0 = u0 * cs.x - u1 * cs.y, o1 = u0 * cs.y + u1 * cs.x;
    if (is_q) {
        float *q = a.q_out + ((long)m * a.nq + h) * a.hd;
        q[i] = o0;
        q[i + half] = o1;
    } else {
        const long slot = a.cap > 0 ? (long)(pos % a.cap) : (long)m;
        float *k = a.k_store + (slot * a.nkv + hk) * a.hd;
        float *v = a.v_store + (slot * a.nkv + hk) * a.hd;
        const int cv = (a.nq + a.nkv + hk) * a.hd;
        k[i] = o0;
        k[i + half] = o1;
        v[i] = val(cv + i);
        v[i + half] = val(cv + i + half);
    }
    stamp_done(a.ps);
}

cudaError_t launch_qk(const QkArgs &a, cudaStream_t s) {
    const int heads = (a.q_out ? a.nq : 0) + (a.k_store ? a.nkv : 0);
    if (heads == 0) return cudaSuccess;
    if (a.hd / 2 < 32 || a.hd / 2 > 1024 || (a.hd / 2) % 32) return cudaErrorInvalidValue;
    return launch_pdl(k_qk, dim3(a.M, heads), dim3(a.hd / 2), 0, s, a);
}

// ---------------------------------------------------------------------------------------------------
// Attention. One thread-block cluster of CL CTAs per unit of HP query heads (HP = 2 when the pass has at
// most 8 rows and a key/value group holds an even number of heads: the two heads fill the 16 rows of
// the tensor-core tile and share every key/value block they load). Keys are cut into blocks of
// kAttnKeys ABSOLUTE positions (block b = positions 32b .. 32b+31); CTA r of the cluster takes the
// blocks b with b % CL == r, in ascending order, and folds each into a running softmax state per
// tile row (max, sum, sum of p*v). The states of the cluster's CTAs are then merged in rank order through
// distributed shared memory. A row's result depends only on its own visible keys and their absolute
// positions (a block with no visible key leaves the state exactly unchanged), so it does not depend on
// how many rows the pass carries or where the pass starts.
// Target (mode 0): row m at position p = n+m sees plane positions max(0, p-window+1)..p (0..p on full
// layers). Draft (mode 1): every row sees context positions max(0, n-window)..n-1, plus all nB keys of
// the block's own store as one extra block after the context blocks.
// ---------------------------------------------------------------------------------------------------
constexpr int kAttnThreads = 512;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnKQ = kAttnWarps / 4;   // parts of the head dimension in the score products
constexpr int kAttnKeys = 32;

// Both products of a block run on the tensor cores (mma.m16n8k16, bf16 in, fp32 accumulate) with every
// fp32 operand split into bf16 hi + lo and the three products hi*hi + hi*lo + lo*hi added (the lo*lo
// term is below fp32 rounding): scores S = Q K^T (16 rows x 32 keys) and O += P V.
//   Scores: warp w takes keys 8*(w%4) .. +7 and part w/4 of kAttnKQ of the head dimension; the parts'
//   partial scores are added in the softmax step (in part order).
//   p.V: warp w takes head-dimension column tiles w + 16t (8 columns each) that exist, all 16 rows, all 32 keys.
// Row pitches (fp32 words): queries and keys hd+8 (fragment loads of 8 rows x 4 column pairs hit 32
// banks), values hd+4 (fragment loads of 4 row pairs x 8 columns hit 32 banks).
constexpr int kAttnKS = 16 / kAttnKQ;   // k-steps of 16 per part of the head dimension (hd <= 256)
constexpr int kAttnNT = 32 / kAttnWarps; // 8-column tiles per warp in p.V (hd <= 256)
constexpr int kAttnSP = 40;  // pitch of the score and probability rows (32 keys + 8)
// key/value blocks in flight (the ring's slots): as many as shared memory holds, so a CTA's blocks are
// requested at once (a CTA takes 1-8 blocks at the step's shapes)
constexpr int attn_buf(int hd) { return hd > 128 ? 3 : 5; }

size_t attn_smem(int hd, int nb) {
    return ((size_t)kMaxRows * (hd + 8) + nb * (size_t)kAttnKeys * (hd + 8) + nb * (size_t)kAttnKeys * (hd + 4) +
            (kAttnKQ + 1) * (size_t)kMaxRows * kAttnSP + 3 * kMaxRows) * 4;
}
size_t attn_smem(int hd) { return attn_smem(hd, attn_buf(hd)); }

template <int N>
__device__ __forceinline__ void cp_async_wait_n() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// fp32 pair -> bf16x2 hi and lo (x = hi + lo to 2^-17 relative), lower element in the low half; the
// roundings are the hardware's paired round-to-nearest-even conversion
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Tile row r holds pass row m = r (HP = 1) or m = r % 8 of head 2u + r / 8 (HP = 2). NB: ring slots.
template <int CL, int HP, int NB>
__global__ void __launch_bounds__(kAttnThreads) k_attn(AttnArgs a) {
    constexpr int kAttnBuf = NB;
    extern __shared__ __align__(16) float sm[];
    const int hd = a.hd, ldq = hd + 8, ldv = hd + 4, hd4 = hd / 4;
    float *Qs = sm;                                 // [16][ldq] this head's query rows
    float *Kb = Qs + kMaxRows * ldq;                // [kAttnBuf][32][ldq] key blocks in flight
    float *Vb = Kb + kAttnBuf * kAttnKeys * ldq;    // [kAttnBuf][32][ldv]
    float *Sp = Vb + kAttnBuf * kAttnKeys * ldv;    // [kAttnKQ][16][kAttnSP] partial scores per part
    float *Ps = Sp + kAttnKQ * kMaxRows * kAttnSP;  // [16][kAttnSP] probabilities of the current block
    float *Sc = Ps + kMaxRows * kAttnSP;            // [16] rescale of the running sums
    float *Mx = Sc + kMaxRows;                      // [16] running max
    float *Ls = Mx + kMaxRows;                      // [16] running sum
    float *Os = Kb;                                 // [16][hd] final state (after the last block)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
    const int unit = blockIdx.x / CL;
    const unsigned rank = cluster_rank();
    const int g = unit * HP / (a.nq / a.nkv);
    auto row_m = [](int r) { return HP == 1 ? r : (r & 7); };
    auto row_h = [unit](int r) { return HP == 1 ? unit : 2 * unit + (r >> 3); };
    // st->n was set before the pass began (every kernel of the pass waits for its predecessor), so it
    // may be read before this kernel's own dependency wait. A pass of more than 16 rows (fp32 output)
    // is cut into tiles of 16 rows along grid y: tile y holds rows 16y.. at positions n + 16y + m.
    const int n_pass = a.st->n;
    const int row_base = kMaxRows * int(blockIdx.y);
    const int n = n_pass + row_base;
    const int M = min(a.M - row_base, kMaxRows);
    int lo, hi;   // inclusive range of plane positions any row may see
    if (a.mode == 0) {
        lo = a.window > 0 ? max(0, n - a.window + 1) : 0;
        hi = n + M - 1;
    } else {
        lo = a.window > 0 ? max(0, n - a.window) : 0;
        hi = n - 1;
    }
    const bool anyA = hi >= lo;
    const int bA0 = anyA ? lo / kAttnKeys : 0, bA1 = anyA ? hi / kAttnKeys : -1;
    const int bV = (a.mode == 1 && a.nB > 0) ? (anyA ? bA1 + 1 : 0) : -1;   // the draft block's own keys
    // this CTA's blocks: b0, b0 + 8, ... <= bA1, then bV when it is ours
    const int b0 = bA0 + int((rank - unsigned(bA0 % CL) + CL) % CL);
    const int nAmine = b0 <= bA1 ? (bA1 - b0) / CL + 1 : 0;
    const int nmine = nAmine + ((bV >= 0 && bV % CL == (int)rank) ? 1 : 0);

    // every warp: keys 4w..4w+3 of the block, 16-byte asynchronous copies by the lanes (rows outside
    // every row's range are zeroed: they are masked, and 0 * v must stay 0); one commit group per block
    auto load_block = [&](int i, int buf) {
        float *K = Kb + buf * kAttnKeys * ldq, *V = Vb + buf * kAttnKeys * ldv;
        const bool virt = i >= nAmine;
        const int b = virt ? bV : b0 + CL * i;
#pragma unroll
        for (int kk = 0; kk < kAttnKeys / kAttnWarps; ++kk) {
            const int j = warp * (kAttnKeys / kAttnWarps) + kk;
            const float *ks = nullptr, *vs = nullptr;
            if (virt) {
                if (j < a.nB) {
                    const long off = ((long)j * a.nkv + g) * hd;
                    ks = a.kB + off;
                    vs = a.vB + off;
                }
            } else {
                const int pos = kAttnKeys * b + j;
                if (pos >= lo && pos <= hi) {
                    const long off = ((long)(pos % a.capA) * a.nkv + g) * hd;
                    ks = a.kA + off;
                    vs = a.vA + off;
                }
            }
            for (int d4 = lane; d4 < hd4; d4 += 32) {
                float *kd = K + j * ldq + 4 * d4, *vd = V + j * ldv + 4 * d4;
                if (ks) {
                    cp_async16(kd, ks + 4 * d4);
                    cp_async16(vd, vs + 4 * d4);
                } else {
                    *reinterpret_cast<float4 *>(kd) = make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4 *>(vd) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
        cp_async_commit();
    };

    // blocks whose positions all precede the pass were written by earlier passes: they are immutable
    // here and are requested before the dependency wait (the pass's own rows come from the kernel
    // before this one)
    auto early = [&](int i) { return a.mode == 0 && i < nAmine && kAttnKeys * (b0 + CL * i) + kAttnKeys <= n_pass; };
    int issued = 0;
    while (issued < kAttnBuf - 1 && issued < nmine && early(issued)) {
        load_block(issued, issued);
        ++issued;
    }
    pdl_wait();
    pdl_trigger();
    stamp_ready(a.ps);
    while (issued < kAttnBuf - 1 && issued < nmine) {
        load_block(issued, issued);
        ++issued;
    }
    for (int k = issued; k < kAttnBuf - 1; ++k) cp_async_commit();   // the prologue is kAttnBuf - 1 groups
    for (int e = tid; e < kMaxRows * hd4; e += kAttnThreads) {
        const int r = e / hd4, d4 = e % hd4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row_m(r) < M)
            v = *reinterpret_cast<const float4 *>(a.q + ((long)(row_base + row_m(r)) * a.nq + row_h(r)) * hd + 4 * d4);
        *reinterpret_cast<float4 *>(Qs + r * ldq + 4 * d4) = v;
    }
    if (tid < kMaxRows) Mx[tid] = -INFINITY, Ls[tid] = 0.f, Sc[tid] = 0.f;
    // tile rows the pass does not carry keep probability 0 and rescale 0 (the softmax step skips them)
    for (int e = tid; e < kMaxRows * kAttnKeys; e += kAttnThreads)
        if (row_m(e / kAttnKeys) >= M) Ps[(e / kAttnKeys) * kAttnSP + e % kAttnKeys] = 0.f;
    __syncthreads();

    // this warp's query fragments (A operand, rows 0..15, its half of the head dimension), hi and lo
    const int kg = warp & 3, kh = warp >> 2;
    const int ksn = hd / (16 * kAttnKQ);           // k-steps per part
    uint32_t qh[kAttnKS][4], ql[kAttnKS][4];
#pragma unroll
    for (int s = 0; s < kAttnKS; ++s) {
        if (s < ksn) {
            const int c = 16 * (kh * ksn + s) + 2 * tq;
            const float2 x0 = *reinterpret_cast<const float2 *>(Qs + gq * ldq + c);
            const float2 x1 = *reinterpret_cast<const float2 *>(Qs + (gq + 8) * ldq + c);
            const float2 x2 = *reinterpret_cast<const float2 *>(Qs + gq * ldq + c + 8);
            const float2 x3 = *reinterpret_cast<const float2 *>(Qs + (gq + 8) * ldq + c + 8);
            split2(x0.x, x0.y, qh[s][0], ql[s][0]);
            split2(x1.x, x1.y, qh[s][1], ql[s][1]);
            split2(x2.x, x2.y, qh[s][2], ql[s][2]);
            split2(x3.x, x3.y, qh[s][3], ql[s][3]);
        }
    }
    // p.V accumulators: tiles nt = warp + kAttnWarps*t (columns 8nt .. 8nt+7), C fragment layout
    const int ntiles = hd / 8;                     // tile nt = warp + kAttnWarps*t exists while nt < ntiles
    float o[kAttnNT][4];
#pragma unroll
    for (int t = 0; t < kAttnNT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;

    for (int i = 0; i < nmine; ++i) {
        const int buf = i % kAttnBuf;
        // keep kAttnBuf - 1 blocks requested ahead (the refilled buffer was released last round). Group
        // j holds block j: the prologue committed kAttnBuf - 1 groups and every round commits one
        // (empty past the end), so block i has landed once at most kAttnBuf - 1 newer groups are pending
        if (issued < nmine) {
            load_block(issued, issued % kAttnBuf);
            ++issued;
        } else {
            cp_async_commit();
        }
        cp_async_wait_n<kAttnBuf - 1>();
        __syncthreads();
        const float *K = Kb + buf * kAttnKeys * ldq, *V = Vb + buf * kAttnKeys * ldv;
        const bool virt = i >= nAmine;
        const int b = virt ? bV : b0 + CL * i;
        // partial scores of this warp's 8 keys over its half of the head dimension
        {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const float *kr = K + (8 * kg + gq) * ldq;
#pragma unroll
            for (int s = 0; s < kAttnKS; ++s) {
                if (s < ksn) {
                    const int col = 16 * (kh * ksn + s) + 2 * tq;
                    const float2 k0 = *reinterpret_cast<const float2 *>(kr + col);
                    const float2 k1 = *reinterpret_cast<const float2 *>(kr + col + 8);
                    uint32_t bh0, bl0, bh1, bl1;
                    split2(k0.x, k0.y, bh0, bl0);
                    split2(k1.x, k1.y, bh1, bl1);
                    mma_bf16(c, qh[s][0], qh[s][1], qh[s][2], qh[s][3], bh0, bh1);
                    mma_bf16(c, qh[s][0], qh[s][1], qh[s][2], qh[s][3], bl0, bl1);
                    mma_bf16(c, ql[s][0], ql[s][1], ql[s][2], ql[s][3], bh0, bh1);
                }
            }
            float *sp = Sp + kh * kMaxRows * kAttnSP;
            *reinterpret_cast<float2 *>(sp + gq * kAttnSP + 8 * kg + 2 * tq) = make_float2(c[0], c[1]);
            *reinterpret_cast<float2 *>(sp + (gq + 8) * kAttnSP + 8 * kg + 2 * tq) = make_float2(c[2], c[3]);
        }
        __syncthreads();
        // softmax update: warp -> rows warp, warp + kAttnWarps, ...; lane -> key
#pragma unroll
        for (int rr = 0; rr < kMaxRows / kAttnWarps; ++rr) {
            const int r = warp + kAttnWarps * rr;
            const int m = row_m(r);
            if (m >= M) continue;
            const int j = lane;
            bool vis;
            if (virt) {
                vis = j < a.nB;
            } else {
                const int pos = kAttnKeys * b + j;
                if (a.mode == 0) {
                    const int p = n + m;
                    vis = pos <= p && (a.window <= 0 || pos > p - a.window) && pos >= 0;
                } else {
                    vis = pos >= lo && pos <= hi;
                }
            }
            float sraw = Sp[r * kAttnSP + j];
#pragma unroll
            for (int part = 1; part < kAttnKQ; ++part) sraw += Sp[(part * kMaxRows + r) * kAttnSP + j];
            const float sv = vis ? sraw * a.scale : -INFINITY;
            float bm = sv;
#pragma unroll
            for (int oo = 16; oo > 0; oo >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, oo));
            const float mo = Mx[r];
            const float mn = fmaxf(mo, bm);
            const float pj = vis ? expf(sv - mn) : 0.f;
            float ps = pj;
#pragma unroll
            for (int oo = 16; oo > 0; oo >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, oo);
            const float sc = mo == -INFINITY ? 0.f : expf(mo - mn);
            Ps[r * kAttnSP + j] = pj;
            __syncwarp();
            if (lane == 0) {
                Sc[r] = sc;
                Mx[r] = mn;
                Ls[r] = fmaf(Ls[r], sc, ps);
            }
        }
        __syncthreads();
        // running p.V over the block's 32 keys (two k-steps of 16)
        {
            const float s0 = Sc[gq], s1 = Sc[gq + 8];
#pragma unroll
            for (int t = 0; t < kAttnNT; ++t) {
                o[t][0] *= s0, o[t][1] *= s0, o[t][2] *= s1, o[t][3] *= s1;
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int kc = 16 * ks + 2 * tq;
                const float2 p0 = *reinterpret_cast<const float2 *>(Ps + gq * kAttnSP + kc);
                const float2 p1 = *reinterpret_cast<const float2 *>(Ps + (gq + 8) * kAttnSP + kc);
                const float2 p2 = *reinterpret_cast<const float2 *>(Ps + gq * kAttnSP + kc + 8);
                const float2 p3 = *reinterpret_cast<const float2 *>(Ps + (gq + 8) * kAttnSP + kc + 8);
                uint32_t ah[4], al[4];
                split2(p0.x, p0.y, ah[0], al[0]);
                split2(p1.x, p1.y, ah[1], al[1]);
                split2(p2.x, p2.y, ah[2], al[2]);
                split2(p3.x, p3.y, ah[3], al[3]);
#pragma unroll
                for (int t = 0; t < kAttnNT; ++t) {
                    if (warp + kAttnWarps * t < ntiles) {
                        const int col = 8 * (warp + kAttnWarps * t) + gq;
                        const float *vr = V + kc * ldv + col;
                        uint32_t bh0, bl0, bh1, bl1;
                        split2(vr[0], vr[ldv], bh0, bl0);
                        split2(vr[8 * ldv], vr[9 * ldv], bh1, bl1);
                        mma_bf16(o[t], ah[0], ah[1], ah[2], ah[3], bh0, bh1);
                        mma_bf16(o[t], ah[0], ah[1], ah[2], ah[3], bl0, bl1);
                        mma_bf16(o[t], al[0], al[1], al[2], al[3], bh0, bh1);
                    }
                }
            }
        }
        __syncthreads();   // the buffer is refilled in the next round
    }
    // publish this CTA's state, then merge the cluster's states in rank order
#pragma unroll
    for (int t = 0; t < kAttnNT; ++t) {
        if (warp + kAttnWarps * t < ntiles) {
            const int col = 8 * (warp + kAttnWarps * t) + 2 * tq;
            if (row_m(gq) < M) *reinterpret_cast<float2 *>(Os + gq * hd + col) = make_float2(o[t][0], o[t][1]);
            if (row_m(gq + 8) < M) *reinterpret_cast<float2 *>(Os + (gq + 8) * hd + col) = make_float2(o[t][2], o[t][3]);
        }
    }
    cluster_sync_all();
    const int ng16 = hd / 16;
    const int items = (HP == 1 ? M : kMaxRows) * ng16;   // (tile row, 16-column group)
    const int hw = tid >> 4;                               // half warp: one item per round
    constexpr int kStride = CL * (kAttnThreads / 16);
    constexpr int kRounds = (kMaxRows * 16 + kStride - 1) / kStride;   // hd <= 256
    float res[kRounds];
    int res_m[kRounds], res_col[kRounds];
    bool res_on[kRounds];
    // every rank's (max, sum, partial output) is requested at once, then combined in rank order
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
        const int it = k * kStride + int(rank) + CL * hw;
        const int r = it / ng16;
        res_on[k] = it < items && row_m(r) < M;
        res[k] = 0.f;
        res_m[k] = res_col[k] = 0;
        if (res_on[k]) {
            const int d = 16 * (it % ng16) + (tid & 15);
            float mr[CL], lr[CL], orr[CL];
#pragma unroll
            for (int q = 0; q < CL; ++q) {
                mr[q] = ld_cluster(Mx + r, q);
                lr[q] = ld_cluster(Ls + r, q);
                orr[q] = ld_cluster(Os + r * hd + d, q);
            }
            float mt = -INFINITY;
#pragma unroll
            for (int q = 0; q < CL; ++q) mt = fmaxf(mt, mr[q]);
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int q = 0; q < CL; ++q) {
                const float f = mr[q] == -INFINITY ? 0.f : expf(mr[q] - mt);
                den = fmaf(lr[q], f, den);
                num = fmaf(orr[q], f, num);
            }
            res[k] = num / den;
            res_m[k] = row_m(r);
            res_col[k] = row_h(r) * hd + d;
        }
    }
    cluster_arrive();   // no reads of other CTAs' shared memory from here on
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
        if (a.out32) {
            if (res_on[k]) a.out32[(long)(row_base + res_m[k]) * (a.nq * hd) + res_col[k]] = res[k];
        } else {
            const float hl = res_on[k] ? act_store(a.outf, a.nq * hd, res_m[k], res_col[k], res[k]) : 0.f;
            const float sg = half_warp_sum(hl);   // every lane of the warp takes part
            if (res_on[k] && (tid & 15) == 0) a.outs[(res_col[k] >> 4) * kMaxRows + res_m[k]] = sg;
        }
    }
    cluster_wait();     // no CTA leaves while another still reads its shared memory
    stamp_done(a.ps);
}

// Cluster size per layer shape: the largest of 16 (a non-portable size), 8 and 4 such that all of the
// shape's clusters fit on the device at once (one wave; a second wave would double the launch). The
// fit is asked once per head-dimension class at context creation, outside any stream capture; until
// then every launch takes clusters of 8. The size depends only on the shape, never on the number of
// rows, so a row's result does not depend on the pass it travels in.
// [device][hd > 128][16, 8]: clusters that fit at once (until attn_prepare: none of 16, all of 8)
static int g_fit[kMaxDevices][2][2];
static bool g_fit_set[kMaxDevices];
template <int CL, int HP, int NB>
static cudaError_t attn_attrs_nb() {
    static bool done[kMaxDevices] = {};
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    const int smem = int(NB == attn_buf(256) ? attn_smem(256, NB) : attn_smem(128, NB));
    cudaError_t e = cudaFuncSetAttribute(k_attn<CL, HP, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess && CL > 8)
        e = cudaFuncSetAttribute(k_attn<CL, HP, NB>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}
template <int CL, int HP>
static cudaError_t attn_attrs() {
    const cudaError_t e = attn_attrs_nb<CL, HP, attn_buf(128)>();
    return e != cudaSuccess ? e : attn_attrs_nb<CL, HP, attn_buf(256)>();
}

template <int CL>
static int clusters_that_fit(int hd) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = attn_smem(hd);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t q = hd > 128 ? cudaOccupancyMaxActiveClusters(&n, k_attn<CL, 2, attn_buf(256)>, &cfg)
                                   : cudaOccupancyMaxActiveClusters(&n, k_attn<CL, 2, attn_buf(128)>, &cfg);
    if (q != cudaSuccess) {
        cudaGetLastError();   // a refused query leaves no sticky error
        n = 0;
    }
    return n;
}

cudaError_t attn_prepare(int hd) {
    cudaError_t e;
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (!g_fit_set[dev]) {
        g_fit[dev][0][0] = g_fit[dev][1][0] = 0;
        g_fit[dev][0][1] = g_fit[dev][1][1] = 1 << 20;
        g_fit_set[dev] = true;
    }
    if ((e = attn_attrs<8, 1>()) || (e = attn_attrs<8, 2>()) || (e = attn_attrs<4, 1>()) || (e = attn_attrs<4, 2>()))
        return e;
    g_fit[dev][hd > 128][1] = clusters_that_fit<8>(hd);
    if (attn_attrs<16, 1>() != cudaSuccess || attn_attrs<16, 2>() != cudaSuccess) {
        cudaGetLastError();   // no wide clusters on this device
        g_fit[dev][hd > 128][0] = 0;
    } else {
        g_fit[dev][hd > 128][0] = clusters_that_fit<16>(hd);
    }
    return cudaSuccess;
}

template <int CL, int HP>
static cudaError_t launch_attn_t(const AttnArgs &a, cudaStream_t s) {
    const cudaError_t e = attn_attrs<CL, HP>();
    if (e != cudaSuccess) return e;
    const int tiles = (a.M + kMaxRows - 1) / kMaxRows;
    const dim3 grid(a.nq / HP * CL, tiles);
    if (a.hd > 128)
        return launch_cluster_pdl(k_attn<CL, HP, attn_buf(256)>, grid, CL, kAttnThreads, attn_smem(a.hd), s, a);
    return launch_cluster_pdl(k_attn<CL, HP, attn_buf(128)>, grid, CL, kAttnThreads, attn_smem(a.hd), s, a);
}

cudaError_t launch_attn(const AttnArgs &a, cudaStream_t s) {
    if (a.hd % 64 || a.hd < 64 || a.hd > 256 || a.M < 1 || (a.M > kMaxRows && (!a.out32 || a.mode != 0)) ||
        a.M > 65535 * kMaxRows || a.nB > kAttnKeys || a.nkv < 1 || a.nq % a.nkv)
        return cudaErrorInvalidValue;
    const bool pairs = (a.nq / a.nkv) % 2 == 0;   // two heads of one key/value group per CTA possible
    const int units = pairs ? a.nq / 2 : a.nq;    // clusters of a pass of up to 8 rows
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    static const int kNoFit[2] = {0, 1 << 20};   // attn_prepare not run on this device: clusters of 8
    const int *fit = g_fit_set[dev] ? g_fit[dev][a.hd > 128] : kNoFit;
    const int cl = (a.max_cluster >= 16 && fit[0] >= units) ? 16 : (a.max_cluster >= 8 && fit[1] >= units) ? 8 : 4;
    const bool hp2 = pairs && a.M <= 8;
    if (cl == 16) return hp2 ? launch_attn_t<16, 2>(a, s) : launch_attn_t<16, 1>(a, s);
    if (cl == 8) return hp2 ? launch_attn_t<8, 2>(a, s) : launch_attn_t<8, 1>(a, s);
    return hp2 ? launch_attn_t<4, 2>(a, s) : launch_attn_t<4, 1>(a, s);
}

// ---------------------------------------------------------------------------------------------------
// The per-layer-embedding tail's two products in one launch: the gate z = silu(x Wg) * p_l (K = H,
// N = P) and the projection y = z Wp (K = P, N = H). One cluster of P/16 CTAs:
//   - CTA r computes the gate's 16-column tile r over all of K: its 8 warps take the 64-input chunks
//     w, w + 8, ... and their sums are added in warp order; then silu * p_l, kept in shared memory.
//   - After a cluster barrier every CTA gathers the whole z (tile r from rank r) into the operand
//     format, then computes its share of the projection's 16-column tiles over all of K = P and
//     writes y's rows (fp32).
// Both weight matrices are requested (cp.async into shared memory) before the dependency wait. The
// Q4_1 math is the product kernel's: codes enter the tensor cores as 128 + q, rows as bf16 hi + lo,
// and each 32-block folds in y += d c + (m - 128 d) S. Every sum has a fixed order, so a row's
// result does not depend on how many rows the pass carries.
// ---------------------------------------------------------------------------------------------------
constexpr int kPleWarps = 8;

__host__ __device__ inline int ple_cluster(int P) { return P / 16; }
__host__ __device__ inline int ple_tiles_per_cta(int H, int P) {
    const int nt = H / 16, cl = ple_cluster(P);
    return (nt + cl - 1) / cl;
}
static size_t ple_smem(int H, int P, int MT) {
    const size_t cg = (size_t)padded_k(H) / 64, cp = (size_t)padded_k(P) / 64, gp = (size_t)padded_k(P) / 16;
    const size_t gh = (size_t)H / 16;
    return cg * 640 + (size_t)ple_tiles_per_cta(H, P) * cp * 640 + MT * gh * 512 + gh * kMaxRows * 4 +
           (size_t)kPleWarps * MT * 4 * 32 * 4 + 16 * 16 * 4 + MT * gp * 512 + gp * kMaxRows * 4;
}

bool ple_fused_ok(int M, int H, int P) {
    return M >= 1 && M <= kMaxRows && P >= 16 && P % 16 == 0 && P / 16 <= 16 && H % 128 == 0 &&
           ple_smem(H, P, M > 8 ? 2 : 1) <= 200 * 1024;
}

// one 64-input chunk of one 16-column tile: codes and (d, m) from `t` (a 640-byte tile in shared
// memory), rows from the operand fragments `xb` (MT row tiles, 4 k-steps) and sums `xsum` (16-input
// groups of the chunk, kMaxRows each); adds into acc
template <int MT>
__device__ __forceinline__ void ple_chunk(float (&acc)[MT][4], const uint8_t *t, const uint4 (&xb)[MT][4],
                                          const float *xsum, int lane) {
    const int g = lane >> 2, tq = lane & 3;
    const uint4 nb = *reinterpret_cast<const uint4 *>(t + 16 * lane);
    const uint4 sc = *reinterpret_cast<const uint4 *>(t + 512 + 16 * g);
    const uint32_t wv[4] = {nb.x, nb.y, nb.z, nb.w};
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        float c[MT][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t w = wv[2 * blk + kk];
            const uint32_t a0 = nib_pair_bf16(w), a1 = nib_pair_bf16(w >> 4), a2 = nib_pair_bf16(w >> 8),
                           a3 = nib_pair_bf16(w >> 12);
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
                const uint4 b = xb[tt][2 * blk + kk];
                if (kk == 0) {
                    c[tt][0] = c[tt][1] = c[tt][2] = c[tt][3] = 0.f;
                }
                mma_bf16(c[tt], a0, a1, a2, a3, b.x, b.y);
                mma_bf16(c[tt], a0, a1, a2, a3, b.z, b.w);
            }
        }
        uint32_t dlo = blk ? sc.z : sc.x, dhi = blk ? sc.w : sc.y;
        const float2 flo = __half22float2(*reinterpret_cast<__half2 *>(&dlo));   // (d, m) of column g
        const float2 fhi = __half22float2(*reinterpret_cast<__half2 *>(&dhi));   // column g + 8
        const float mlo = fmaf(-128.f, flo.x, flo.y), mhi = fmaf(-128.f, fhi.x, fhi.y);
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
            const float *s0 = xsum + (2 * blk) * kMaxRows + 8 * tt + 2 * tq;
            const float *s1 = xsum + (2 * blk + 1) * kMaxRows + 8 * tt + 2 * tq;
            const float S0 = s0[0] + s1[0], S1 = s0[1] + s1[1];
            acc[tt][0] = fmaf(mlo, S0, fmaf(flo.x, c[tt][0], acc[tt][0]));
            acc[tt][1] = fmaf(mlo, S1, fmaf(flo.x, c[tt][1], acc[tt][1]));
            acc[tt][2] = fmaf(mhi, S0, fmaf(fhi.x, c[tt][2], acc[tt][2]));
            acc[tt][3] = fmaf(mhi, S1, fmaf(fhi.x, c[tt][3], acc[tt][3]));
        }
    }
}

template <int MT>
__global__ void __launch_bounds__(kPleWarps * 32) k_ple(PleArgs a) {
    extern __shared__ __align__(16) uint8_t sm8[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
    const unsigned rank = cluster_rank();
    const int CL = ple_cluster(a.P);
    const int Cg = padded_k(a.H) / 64, Cp = padded_k(a.P) / 64, Gp = padded_k(a.P) / 16, G = a.P / 16;
    const int NT = a.H / 16, tpc = ple_tiles_per_cta(a.H, a.P);
    const int t0 = min(NT, int(rank) * tpc), t1 = min(NT, t0 + tpc);
    uint8_t *wg = sm8;                                              // [Cg][640] gate tile `rank`
    uint8_t *wp = wg + (size_t)Cg * 640;                            // [t1 - t0][Cp][640] projection tiles
    uint32_t *xa = reinterpret_cast<uint32_t *>(wp + (size_t)tpc * Cp * 640);   // [MT][H/16][128] gate input
    float *xas = reinterpret_cast<float *>(xa + (size_t)MT * (a.H / 16) * 128);   // [H/16][kMaxRows] its sums
    float *red = xas + (size_t)(a.H / 16) * kMaxRows;               // [warp][tt][4][32]
    float *zs = red + kPleWarps * MT * 4 * 32;                      // [16 rows][16 columns]
    uint32_t *xo = reinterpret_cast<uint32_t *>(zs + 16 * 16);      // [MT][Gp][128 words] operand format
    float *xos = reinterpret_cast<float *>(xo + (size_t)MT * Gp * 128);   // [Gp][kMaxRows] sums

    // weights are immutable: requested before the dependency wait
    {
        const uint8_t *src = a.img_g + (size_t)rank * Cg * 640;
        for (int e = threadIdx.x; e < Cg * 40; e += blockDim.x) cp_async16(wg + 16 * e, src + 16 * e);
        const uint8_t *srp = a.img_p + (size_t)t0 * Cp * 640;
        for (int e = threadIdx.x; e < (t1 - t0) * Cp * 40; e += blockDim.x) cp_async16(wp + 16 * e, srp + 16 * e);
        cp_async_commit();
    }
    pdl_trigger();
    pdl_wait();
    stamp_ready(a.ps);
    // the gate's input rows (all of K: each row block is one run of the operand format) and their sums
    {
        const int nx = MT * (a.H / 16) * 32, ns = (a.H / 16) * kMaxRows / 4;
        for (int e = threadIdx.x; e < nx; e += blockDim.x) cp_async16(xa + 4 * e, a.xf + 4 * e);
        for (int e = threadIdx.x; e < ns; e += blockDim.x) cp_async16(xas + 4 * e, a.xs + 4 * e);
        cp_async_commit();
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- gate: tile `rank`, chunks split over the warps ----
    float acc[MT][4];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) acc[tt][0] = acc[tt][1] = acc[tt][2] = acc[tt][3] = 0.f;
    for (int c = warp; c < Cg; c += kPleWarps) {
        uint4 xb[MT][4];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                xb[tt][ks] = *reinterpret_cast<const uint4 *>(xa + act_group(a.H, 8 * tt, 4 * c + ks) + 4 * lane);
        ple_chunk<MT>(acc, wg + (size_t)c * 640, xb, xas + (size_t)(4 * c) * kMaxRows, lane);
    }
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[((warp * MT + tt) * 4 + i) * 32 + lane] = acc[tt][i];
    __syncthreads();
    // sum over warps in order, then z = silu(.) * p_l; rows past M are zero
    for (int e = threadIdx.x; e < 16 * 16; e += blockDim.x) {
        const int tok = e >> 4, col = e & 15;
        float z = 0.f;
        if (tok < 8 * MT) {
            const int tt = tok >> 3, i = (col >= 8 ? 2 : 0) + (tok & 1), ln = 4 * (col & 7) + ((tok & 7) >> 1);
            float v = 0.f;
            for (int w = 0; w < kPleWarps; ++w) v += red[((w * MT + tt) * 4 + i) * 32 + ln];
            if (tok < a.M) z = silu_f(v) * bf16_to_f32(a.ext[(long)tok * a.lde + 16 * rank + col]);
        }
        zs[e] = z;
    }
    cluster_sync_all();   // every rank's tile of z is in its shared memory

    // ---- the projection's input: z in operand format (group kb from rank kb), zero past P ----
    for (int e = threadIdx.x; e < MT * Gp * 32; e += blockDim.x) {
        const int ln = e & 31, kb = (e >> 5) % Gp, tt = (e >> 5) / Gp;
        const int gg = ln >> 2, t = ln & 3, tok = 8 * tt + gg;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (kb < G) {
            const int cols[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = ld_cluster(zs + tok * 16 + cols[q], unsigned(kb));
        }
        uint32_t hi[2], lo[2];
        float hl = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
            const float2 hf = __bfloat1622float2(h);
            const __nv_bfloat162 l = __floats2bfloat162_rn(v[2 * q] - hf.x, v[2 * q + 1] - hf.y);
            const float2 lf = __bfloat1622float2(l);
            hi[q] = *reinterpret_cast<const uint32_t *>(&h);
            lo[q] = *reinterpret_cast<const uint32_t *>(&l);
            hl += (hf.x + lf.x) + (hf.y + lf.y);
        }
        *reinterpret_cast<uint4 *>(xo + ((size_t)tt * Gp + kb) * 128 + 4 * ln) = make_uint4(hi[0], hi[1], lo[0], lo[1]);
        // the row's 16-input sum: the four lanes t of row gg hold its four entries
        hl += __shfl_xor_sync(0xffffffffu, hl, 1);
        hl += __shfl_xor_sync(0xffffffffu, hl, 2);
        if (t == 0) xos[kb * kMaxRows + tok] = hl;
    }
    cluster_arrive();   // no more reads of other ranks' shared memory
    __syncthreads();

    // ---- projection: this rank's tiles t0..t1-1 in pairs, all of K = P per warp ----
    for (int p0 = t0 + 2 * warp; p0 < t1; p0 += 2 * kPleWarps) {
        float ac[2][MT][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) ac[j][tt][0] = ac[j][tt][1] = ac[j][tt][2] = ac[j][tt][3] = 0.f;
        const bool two = p0 + 1 < t1;
        for (int c = 0; c < Cp; ++c) {
            uint4 xb[MT][4];
#pragma unroll
            for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    xb[tt][ks] = *reinterpret_cast<const uint4 *>(xo + ((size_t)tt * Gp + 4 * c + ks) * 128 + 4 * lane);
            const float *xsum = xos + (size_t)(4 * c) * kMaxRows;
            ple_chunk<MT>(ac[0], wp + ((size_t)(p0 - t0) * Cp + c) * 640, xb, xsum, lane);
            if (two) ple_chunk<MT>(ac[1], wp + ((size_t)(p0 + 1 - t0) * Cp + c) * 640, xb, xsum, lane);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (j == 1 && !two) break;
            const int tile = p0 + j;
#pragma unroll
            for (int tt = 0; tt < MT; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = 8 * tt + 2 * tq + (i & 1), col = 16 * tile + g + 8 * (i >> 1);
                    if (tok < a.M) a.y[(long)tok * a.H + col] = ac[j][tt][i];
                }
        }
    }
    cluster_wait();   // no rank leaves while another may still read its tile of z
    stamp_done(a.ps);
}

template <int MT>
static cudaError_t launch_ple_t(const PleArgs &a, cudaStream_t s) {
    static bool done[kMaxDevices] = {};
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    const size_t smem = ple_smem(a.H, a.P, MT);
    if (!done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_ple<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k_ple<MT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    const int cl = ple_cluster(a.P);
    return launch_cluster_pdl(k_ple<MT>, dim3(cl), cl, kPleWarps * 32, smem, s, a);
}

cudaError_t launch_ple(const PleArgs &a, cudaStream_t s) {
    if (!ple_fused_ok(a.M, a.H, a.P)) return cudaErrorInvalidValue;
    return a.M > 8 ? launch_ple_t<2>(a, s) : launch_ple_t<1>(a, s);
}

// ---------------------------------------------------------------------------------------------------
// Elementwise steps of a long pass on fp32 rows (a pass of 16 rows or fewer runs them in the products'
// epilogues): the FFN's gate, and the per-layer-embedding gate.
// four consecutive outputs per thread (F is a multiple of 64)
__global__ void k_glu32(const float *__restrict__ y, int M, int F, float *__restrict__ out) {
    const long i = blockIdx.x * (long)blockDim.x + threadIdx.x;   // index of a group of four outputs
    const int F4 = F / 4;
    if (i >= (long)M * F4) return;
    const long m = i / F4;
    const int j = int(i % F4) * 4;
    const float4 g = *reinterpret_cast<const float4 *>(y + m * 2 * F + j);
    const float4 u = *reinterpret_cast<const float4 *>(y + m * 2 * F + F + j);
    *reinterpret_cast<float4 *>(out + m * F + j) =
        make_float4(silu_f(g.x) * u.x, silu_f(g.y) * u.y, silu_f(g.z) * u.z, silu_f(g.w) * u.w);
}

__global__ void k_silu_mul32(const float *__restrict__ y, int M, int P, const uint16_t *__restrict__ e, int lde,
                             float *__restrict__ out) {
    const long i = blockIdx.x * (long)blockDim.x + threadIdx.x;
    if (i >= (long)M * P) return;
    const long m = i / P;
    const int j = int(i % P);
    out[i] = silu_f(y[i]) * bf16_to_f32(e[m * lde + j]);
}

cudaError_t launch_glu32(const float *y, int M, int F, float *out, cudaStream_t s) {
    if (F % 4) return cudaErrorInvalidValue;
    const long n = (long)M * (F / 4);
    k_glu32<<<unsigned((n + 255) / 256), 256, 0, s>>>(y, M, F, out);
    return cudaGetLastError();
}

cudaError_t launch_silu_mul32(const float *y, int M, int P, const uint16_t *e, int lde, float *out, cudaStream_t s) {
    const long n = (long)M * P;
    k_silu_mul32<<<unsigned((n + 255) / 256), 256, 0, s>>>(y, M, P, e, lde, out);
    return cudaGetLastError();
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
    pdl_trigger();
    pdl_wait();
    __shared__ float redf[33];
    __shared__ double wsum[32];
    __shared__ int s_tok, s_last;
    stamp_ready(a.ps);
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
    const int pos = a.st->n + a.row0 + m + 1;
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
    stamp_done(a.ps);
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
    pdl_trigger();
    pdl_wait();
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
