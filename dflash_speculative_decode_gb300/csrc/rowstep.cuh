// rowstep.cuh -- the residual row step (x += RMSNorm(y) w, x *= lambda, tap, next norm in operand format)
// and the q/k step (q/k RMSNorm, rotary embedding, KV store) as device functions, shared by the row and
// q/k kernels and by the products that finish these steps on their own last CTAs.
#pragma once

#include "common.cuh"

namespace dfl {

// Loads of values other CTAs wrote (cache-global, from L2), predicated: 0 when !ok. They are volatile
// asm, so a batch of them goes out in program order before the first of them is used.
__device__ __forceinline__ float2 ldcg2_if(const float *p, bool ok) {
    float2 v;
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %3, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\t"
        "@q ld.global.cg.v2.f32 {%0, %1}, [%2];\n\t}"
        : "=f"(v.x), "=f"(v.y)
        : "l"(p), "r"(int(ok)));
    return v;
}
__device__ __forceinline__ float ldcg_if(const float *p, bool ok) {
    float v;
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\tmov.b32 %0, 0;\n\t@q ld.global.cg.f32 %0, [%1];\n\t}"
                 : "=f"(v)
                 : "l"(p), "r"(int(ok)));
    return v;
}

// two consecutive bf16 weights
__device__ __forceinline__ float2 bf16x2(const uint16_t *w) {
    const uint32_t u = *reinterpret_cast<const uint32_t *>(w);
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// segments of the quad that holds column c of an EPI_PART product, and the first segment's address of
// (row m, column c)
__device__ __forceinline__ int part_nseg(const PartView &v, int c) {
    const int q = c >> 7;
    const long qa = (long)q * v.C;
    return int(cta_of(qa + v.C - 1, v.U, v.G) - cta_of(qa, v.U, v.G)) + 1;
}
__device__ __forceinline__ const float *part_at(const PartView &v, int m, int c) {
    return v.part + ((size_t)(c >> 5) * v.maxseg * kMaxRows + m) * 32 + (c & 31);
}
constexpr size_t kPartSegStride = (size_t)kMaxRows * 32;   // floats between segments

// block-wide sum of four values at once (fixed order, as block_sum)
__device__ __forceinline__ float4 block_sum4(float4 v, float4 *red4) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v.x = warp_sum(v.x), v.y = warp_sum(v.y), v.z = warp_sum(v.z), v.w = warp_sum(v.w);
    if (lane == 0) red4[w] = v;
    __syncthreads();
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (w == 0) {
        t = lane < nw ? red4[lane] : t;
        t.x = warp_sum(t.x), t.y = warp_sum(t.y), t.z = warp_sum(t.z), t.w = warp_sum(t.w);
        if (lane == 0) red4[32] = t;
    }
    __syncthreads();
    return red4[32];
}

// Column groups per thread of the row step that products run on their last CTAs (288 threads): rows of
// up to 12 * 288 = 3456 columns. Wider rows take the separate row kernel.
constexpr int kProductRowPer = 3;
constexpr int kProductRowThreads = 288;   // threads of a product CTA
constexpr int kProductRowCols = 4 * kProductRowPer * kProductRowThreads;

// Slot j of a row of H columns (j < H/4): 16-input group kb = j / 4, lane column t = j % 4, the columns
// ca = 16 kb + 2 t, ca + 1, ca + 8, ca + 9 -- the four inputs whose bf16 hi and lo halves make one
// 16-byte word of the operand format (word act_group(H, row, kb) + 4 t), so a slot's output is a single
// store and four consecutive slots write 64 contiguous bytes. Thread t of the CTA takes the slots
// t + i * blockDim.x (i < PER); blockDim.x is a multiple of 32, so the four slots of a group sit in
// consecutive lanes.
__device__ __forceinline__ int slot_col(int j) { return 16 * (j >> 2) + 2 * (j & 3); }

// the norm weights of the calling thread's slots (see row_step)
template <int PER>
__device__ __forceinline__ void row_weights(const RowArgs &a, float4 (&wp)[PER], float4 (&wn)[PER]) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int j = int(threadIdx.x) + i * int(blockDim.x), ca = slot_col(j);
        const bool on = 4 * j < a.H;
        float2 p0 = make_float2(0.f, 0.f), p1 = p0, n0 = p0, n1 = p0;
        if (on && a.w_post) p0 = bf16x2(a.w_post + ca), p1 = bf16x2(a.w_post + ca + 8);
        if (on && a.w_next) n0 = bf16x2(a.w_next + ca), n1 = bf16x2(a.w_next + ca + 8);
        wp[i] = make_float4(p0.x, p0.y, p1.x, p1.y);
        wn[i] = make_float4(n0.x, n0.y, n1.x, n1.y);
    }
}

// The row step of row m, by every thread of the calling CTA (blockDim a multiple of 32, at most 1024):
//   x += RMSNorm(y, w_post) (or x += y), x *= lambda, tap = x, out = RMSNorm(x, w_next) in operand format.
// y is the product's row: the sum of its segment partials in segment order (or plain rows). wp / wn are
// the norm weights of the thread's slots (loaded by the caller, so their latency can hide behind a wait).
// Every load of the thread's columns goes out in one batch before any is used. The row sums are block
// sums in a fixed order: the result does not depend on how many rows the pass carries.
// NSB: segments of each slot in the batch (more are added after it, in order).
template <int PER, int NSB = 8>
__device__ __forceinline__ void row_step(const RowArgs &a, int m, const float4 (&wp)[PER], const float4 (&wn)[PER],
                                         float *red, float4 *red4) {
    const bool live = !a.rows_from_ctx || m < a.st->ctx_rows;
    float *xr = a.x ? a.x + (long)m * a.H : nullptr;
    const bool have_y = a.yp.part || a.y;
    float2 xa[PER], xb[PER], la[PER][NSB], lb[PER][NSB];
    float4 x[PER], y[PER];
    int ns[PER], ca[PER];
    bool on[PER];
    const float *pp[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int j = int(threadIdx.x) + i * int(blockDim.x);
        on[i] = 4 * j < a.H;
        ca[i] = slot_col(j);
        xa[i] = ldcg2_if(xr + ca[i], on[i] && xr);
        xb[i] = ldcg2_if(xr + ca[i] + 8, on[i] && xr);
        ns[i] = 0;
        pp[i] = nullptr;
        if (on[i] && a.yp.part) {
            ns[i] = part_nseg(a.yp, ca[i]);
            pp[i] = part_at(a.yp, m, ca[i]);
        }
#pragma unroll
        for (int s = 0; s < NSB; ++s) {
            la[i][s] = ldcg2_if(pp[i] + s * kPartSegStride, s < ns[i]);
            lb[i][s] = ldcg2_if(pp[i] + s * kPartSegStride + 8, s < ns[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        x[i] = make_float4(xa[i].x, xa[i].y, xb[i].x, xb[i].y);
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        if (pp[i]) {
#pragma unroll
            for (int s = 0; s < NSB; ++s)
                if (s < ns[i]) t.x += la[i][s].x, t.y += la[i][s].y, t.z += lb[i][s].x, t.w += lb[i][s].y;
            for (int s = NSB; s < ns[i]; ++s) {
                const float2 e0 = ldcg2_if(pp[i] + s * kPartSegStride, true);
                const float2 e1 = ldcg2_if(pp[i] + s * kPartSegStride + 8, true);
                t.x += e0.x, t.y += e0.y, t.z += e1.x, t.w += e1.y;
            }
        } else if (on[i] && a.y) {
            const float *yr = a.y + (long)m * a.ldy + ca[i];
            t = make_float4(yr[0], yr[1], yr[8], yr[9]);
        }
        y[i] = t;
    }
    // With a post-norm, the output norm's sum of squares is expanded so one block reduction gives both:
    //   x' = lambda (x + r y w),  sum x'^2 = lambda^2 (sum x^2 + 2 r sum x y w + r^2 sum (y w)^2),
    //   r = (sum y^2 / H + eps)^(-1/2).
    float r_next = -1.f;   // the output norm's scale when it came out of the combined reduction
    if (have_y) {
        if (a.w_post) {
            float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const float4 w = wp[i], yy = y[i], xx = x[i];
                const float4 yw = make_float4(yy.x * w.x, yy.y * w.y, yy.z * w.z, yy.w * w.w);
                v4.x += (yy.x * yy.x + yy.y * yy.y) + (yy.z * yy.z + yy.w * yy.w);
                v4.y += (xx.x * xx.x + xx.y * xx.y) + (xx.z * xx.z + xx.w * xx.w);
                v4.z += (xx.x * yw.x + xx.y * yw.y) + (xx.z * yw.z + xx.w * yw.w);
                v4.w += (yw.x * yw.x + yw.y * yw.y) + (yw.z * yw.z + yw.w * yw.w);
            }
            v4 = block_sum4(v4, red4);
            const float r = 1.0f / sqrtf(v4.x / a.H + a.eps);
#pragma unroll
            for (int i = 0; i < PER; ++i)
                if (on[i]) {
                    const float4 w = wp[i];
                    x[i].x += (y[i].x * r) * w.x, x[i].y += (y[i].y * r) * w.y;
                    x[i].z += (y[i].z * r) * w.z, x[i].w += (y[i].w * r) * w.w;
                }
            if (a.w_next) {
                const float ss = a.lambda * a.lambda * (v4.y + 2.f * r * v4.z + r * r * v4.w);
                r_next = 1.0f / sqrtf(fmaxf(ss, 0.f) / a.H + a.eps);
            }
        } else {
#pragma unroll
            for (int i = 0; i < PER; ++i) x[i].x += y[i].x, x[i].y += y[i].y, x[i].z += y[i].z, x[i].w += y[i].w;
        }
    }
    float xs = 0.f;
    const int pos = (a.pos_from_ctx ? a.st->draft_n : a.st->n) + m;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        if (a.lambda != 1.0f) x[i].x *= a.lambda, x[i].y *= a.lambda, x[i].z *= a.lambda, x[i].w *= a.lambda;
        if (on[i]) {
            auto put = [&](float *base) {
                *reinterpret_cast<float2 *>(base + ca[i]) = make_float2(x[i].x, x[i].y);
                *reinterpret_cast<float2 *>(base + ca[i] + 8) = make_float2(x[i].z, x[i].w);
            };
            if (xr && (have_y || a.lambda != 1.0f)) put(xr);
            if (a.tap && live) put(a.tap + (long)pos * a.ld_tap + a.tap_off);
            if (a.y_out && have_y) {
                float *yo = a.y_out + (long)m * a.H;
                *reinterpret_cast<float2 *>(yo + ca[i]) = make_float2(y[i].x, y[i].y);
                *reinterpret_cast<float2 *>(yo + ca[i] + 8) = make_float2(y[i].z, y[i].w);
            }
        }
        xs += (x[i].x * x[i].x + x[i].y * x[i].y) + (x[i].z * x[i].z + x[i].w * x[i].w);
    }
    if (a.out32) {
        float r = 1.f;
        if (a.w_next) r = r_next >= 0.f ? r_next : 1.0f / sqrtf(block_sum(xs, red) / a.H + a.eps);
        float *o = a.out32 + (long)m * a.H;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            if (!on[i]) continue;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live) {
                if (a.w_next) {
                    const float4 w = wn[i];
                    v = make_float4((x[i].x * r) * w.x, (x[i].y * r) * w.y, (x[i].z * r) * w.z, (x[i].w * r) * w.w);
                } else {
                    v = x[i];
                }
            }
            *reinterpret_cast<float2 *>(o + ca[i]) = make_float2(v.x, v.y);
            *reinterpret_cast<float2 *>(o + ca[i] + 8) = make_float2(v.z, v.w);
        }
    } else if (a.outf) {
        float r = 1.f;
        if (a.w_next) r = r_next >= 0.f ? r_next : 1.0f / sqrtf(block_sum(xs, red) / a.H + a.eps);
        const int row = a.out_row0 + m;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int j = int(threadIdx.x) + i * int(blockDim.x);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (on[i] && live) {
                if (a.w_next) {
                    const float4 w = wn[i];
                    v = make_float4((x[i].x * r) * w.x, (x[i].y * r) * w.y, (x[i].z * r) * w.z, (x[i].w * r) * w.w);
                } else {
                    v = x[i];
                }
            }
            // hi = bf16(v), lo = bf16(v - hi): {hi(ca, ca+1), hi(ca+8, ca+9), lo(ca, ca+1), lo(ca+8, ca+9)}
            const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
            const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
            const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
            const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
            const float2 g0 = __bfloat1622float2(l0), g1 = __bfloat1622float2(l1);
            float hl = ((f0.x + g0.x) + (f0.y + g0.y)) + ((f1.x + g1.x) + (f1.y + g1.y));
            if (on[i])
                *reinterpret_cast<uint4 *>(a.outf + act_group(a.H, row, j >> 2) + 4 * (j & 3)) =
                    make_uint4(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                               *reinterpret_cast<const uint32_t *>(&l0), *reinterpret_cast<const uint32_t *>(&l1));
            // the four slots of a 16-input group are consecutive lanes
            hl += __shfl_xor_sync(0xffffffffu, hl, 1);
            hl += __shfl_xor_sync(0xffffffffu, hl, 2);
            if (on[i] && (j & 3) == 0) a.outs[(j >> 2) * kMaxRows + row] = hl;
        }
    }
}

// Tasks of a q/k step per row: the query heads (when q_out is set), then for every key-value head a key
// task (norm, rotation, store) and a value task (store).
__host__ __device__ __forceinline__ int qk_heads(const QkArgs &a) {
    return (a.q_out ? a.nq : 0) + (a.k_store ? 2 * a.nkv : 0);
}

// Task h of row m of a q/k step, by one warp. Query and key tasks: RMSNorm over the head dimension, then
// the half-split rotary embedding at the row's absolute position; a query goes to q_out, a key to its
// plane slot (pos mod cap, or the row of a block store). Value tasks store the head's values there.
// Lane l takes the pairs (i, i + hd/2), i = l + 32 jj; all their segments are loaded in one batch and
// added in segment order; the sum of squares is a warp sum in a fixed order.
__device__ __forceinline__ void qk_task(const QkArgs &a, int m, int h, int lane) {
    if (a.live_from_ctx && m >= a.st->ctx_rows) return;
    const int half = a.hd / 2, np = half / 32;   // 1, 2 or 4 pairs per lane
    const int pos = (a.pos_mode == 2 ? a.st->draft_n : a.st->n) + m;
    const int rr = a.row0 + m;
    const int nqh = a.q_out ? a.nq : 0;
    const int kind = h < nqh ? 0 : ((h - nqh) & 1) ? 2 : 1;   // 0 query, 1 key, 2 value
    const int hk = kind == 0 ? 0 : (h - nqh) >> 1;
    const int c0 = kind == 0 ? h * a.hd : kind == 1 ? (a.nq + hk) * a.hd : (a.nq + a.nkv + hk) * a.hd;
    constexpr int NSB = 8;
    float l[8][NSB], u[8];
    int ns[8];
    const float *pc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c = c0 + lane + 32 * (j >> 1) + (j & 1) * half;
        const bool on = (j >> 1) < np;
        ns[j] = 0;
        pc[j] = nullptr;
        u[j] = 0.f;
        if (on && a.qp.part) {
            ns[j] = part_nseg(a.qp, c);
            pc[j] = part_at(a.qp, rr, c);
        } else if (on) {
            u[j] = a.qkv[(long)rr * a.ldq + c];
        }
#pragma unroll
        for (int s = 0; s < NSB; ++s) l[j][s] = ldcg_if(pc[j] + s * kPartSegStride, s < ns[j]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (!pc[j]) continue;
        float t = 0.f;
#pragma unroll
        for (int s = 0; s < NSB; ++s)
            if (s < ns[j]) t += l[j][s];
        for (int s = NSB; s < ns[j]; ++s) t += ldcg_if(pc[j] + s * kPartSegStride, true);
        u[j] = t;
    }
    if (a.qkv_out)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if ((j >> 1) < np) a.qkv_out[(long)rr * a.ldq + c0 + lane + 32 * (j >> 1) + (j & 1) * half] = u[j];
    const long slot = a.cap > 0 ? (long)(pos % a.cap) : (long)m;
    if (kind == 2) {
        float *v = a.v_store + (slot * a.nkv + hk) * a.hd;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            if (jj < np) {
                const int i = lane + 32 * jj;
                v[i] = u[2 * jj];
                v[i + half] = u[2 * jj + 1];
            }
        return;
    }
    const uint16_t *w = kind == 0 ? a.q_norm : a.k_norm;
    float ss = 0.f;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
        if (jj < np) ss += u[2 * jj] * u[2 * jj] + u[2 * jj + 1] * u[2 * jj + 1];
    const float r = 1.0f / sqrtf(warp_sum(ss) / a.hd + a.eps);
    float *dst = kind == 0 ? a.q_out + ((long)m * a.nq + h) * a.hd : a.k_store + (slot * a.nkv + hk) * a.hd;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
        if (jj < np) {
            const int i = lane + 32 * jj;
            const float x0 = (u[2 * jj] * r) * bf16_to_f32(w[i]), x1 = (u[2 * jj + 1] * r) * bf16_to_f32(w[i + half]);
            const float2 cs = a.rope[(long)pos * half + i];
            dst[i] = x0 * cs.x - x1 * cs.y;
            dst[i + half] = x0 * cs.y + x1 * cs.x;
        }
}

}  // namespace dfl
