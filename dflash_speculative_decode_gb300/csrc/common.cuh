// common.cuh -- device helpers and kernel interfaces shared by the library's own CUDA sources.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dfl {

constexpr int kMaxRows = 16;           // rows of one pass (R_max)
constexpr int kWarpsPerCta = 8;        // head CTA: 8 warps, each a range of 16-column tiles

// Device-resident counters of the current pass. The host writes them with k_set_state before each
// pass so a captured graph replays at any position.
struct DevState {
    int n;                 // positions held (committed) at the start of the pass
    int k;                 // rows of this pass
    int draft_n;           // positions whose taps are already draft context
    int ctx_rows;          // committed rows this draft pass makes context (draft_n .. draft_n+ctx_rows-1)
    int accepted;          // accepted length of the last verify
    int sampled;           // 1: sample with temperature, 0: greedy
    float temperature;
    int pad0;
    unsigned long long seed;
    int rows[kMaxRows];    // tokens of the verify rows (row 0 = last token)
    int target[kMaxRows];  // target token per verify row
    int props[kMaxRows];   // draft proposals for positions n+1..n+block-1
    int last_tok;          // row 0 of the last draft block
    int err;               // sticky device-side error bits
};

// DevState::err bits
constexpr int kErrWaitTimeout = 1;   // a bounded wait in a kernel gave up

struct SetStateArgs {
    int n, k, draft_n, ctx_rows, sampled, use_draft_rows, last_tok;
    float temperature;
    unsigned long long seed;
    int rows[kMaxRows];
};

// Function attributes (shared-memory size, cluster sizes) are set once per device.
constexpr int kMaxDevices = 64;
inline int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
    return d;
}

// ---- small device helpers ------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Round to nearest even bf16 (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    const __nv_bfloat16 h = __float2bfloat16_rn(f);   // the hardware conversion (round to nearest even)
    return *reinterpret_cast<const uint16_t *>(&h);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// D = A * B + D for one m16n8k16 bf16 tile, fp32 accumulate. Not volatile: it has no effect beyond its
// outputs, so the compiler may interleave independent products (callers also issue them so that
// consecutive products feed different accumulators).
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two 4-bit codes of a packed word -> a bf16x2 register holding 128 + q exactly: bits [0, 4) and
// [16, 20) of w become the low and high bf16. 0x4300 is bf16 128.0, whose last mantissa bit is worth 1,
// so (0x4300 | q) is 128 + q. A product over such codes carries 128 * sum(x), which the Q4_1 minimum
// term takes back (m - 128 d).
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t w) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may start
// while its predecessor is still running. Everything before pdl_wait() must touch only data no earlier
// kernel writes (weights); pdl_wait() returns once the predecessor grid has completed and its writes are
// visible. pdl_trigger() lets the successor be scheduled (once every CTA of this grid has triggered or
// exited); it orders no memory, so the small row kernels trigger on entry, which lets the product after
// them land on the SMs and stream its first weights while they run. Both are no-ops for a kernel
// launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16-byte asynchronous global -> shared copy (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most one committed group of this thread is still in flight
__device__ __forceinline__ void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_group2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// ---- profiling stamps ---------------------------------------------------------------------------------
// A profiled pass gives each instrumented launch a slot. Thread 0 of every CTA lowers prof[slot] to the
// time it passed its dependency wait and raises prof[kProfSlots + slot] to the time the CTA finished
// (device globaltimer, ns). The launch's in-pass duration is the difference: it excludes the time its
// CTAs spent resident before their dependency was met, so durations of consecutive launches do not
// overlap and add up to no more than the pass. prof == nullptr (not profiling) records nothing.
constexpr int kProfSlots = 2048;
struct Stamp {
    unsigned long long *prof;
    int slot;
};
__device__ __forceinline__ unsigned long long globaltimer_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void stamp_ready(const Stamp &s) {
    if (s.prof && threadIdx.x == 0) atomicMin(s.prof + s.slot, globaltimer_now());
}
// every thread of the CTA calls it (it synchronises the CTA first)
__device__ __forceinline__ void stamp_done(const Stamp &s) {
    if (!s.prof) return;
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(s.prof + kProfSlots + s.slot, globaltimer_now());
}

// ---- activation operand format ---------------------------------------------------------------------
// An activation matrix of up to 16 rows and K inputs (K % 16 == 0) that feeds a product is stored as
// the B fragments of mma.m16n8k16: fp32 x = hi + lo with hi = bf16(x), lo = bf16(x - hi) (exact to
// 2^-17 relative). Rows come in blocks of 8 (rb = tok / 8); for each 16-input group kb the block's 8
// rows are adjacent, 64 bytes each, so a run of groups of one row block is contiguous (one copy per row
// block for a range of inputs). Row tok, group kb, lane column t = 0..3 own 16 bytes at word
// ((rb * K/16 + kb) * 8 + tok % 8) * 16 + t * 4: {hi(2t, 2t+1), hi(2t+8, 2t+9), lo(2t, 2t+1),
// lo(2t+8, 2t+9)}, inputs counted within the group, the lower input in the low half. Beside it,
// sums[kb * 16 + tok] holds the fp32 sum of hi + lo over the row's 16 inputs of group kb (the Q4_1
// minimum term); the product then computes exactly sum_k (hi_k + lo_k) w_k.
// act_group gives the first word of (row tok, group kb); act_store writes one element and returns hi + lo.
__host__ __device__ __forceinline__ long act_group(int K, int tok, int kb) {
    return (((long)(tok >> 3) * (K >> 4) + kb) * 8 + (tok & 7)) * 16;
}
__device__ __forceinline__ float act_store(uint32_t *f, int K, int tok, int k, float v) {
    const int r = k & 15, t = (r & 7) >> 1, w = r >> 3, half = r & 1;
    uint16_t *p = reinterpret_cast<uint16_t *>(f + act_group(K, tok, k >> 4) + t * 4);
    const uint16_t hi = f32_to_bf16(v);
    const uint16_t lo = f32_to_bf16(v - bf16_to_f32(hi));
    p[2 * w + half] = hi;
    p[2 * (w + 2) + half] = lo;
    return bf16_to_f32(hi) + bf16_to_f32(lo);
}

// ---- mbarriers and bulk asynchronous copies ----------------------------------------------------------
constexpr unsigned kWaitHintNs = 20000;              // suspend-time hint of one test (20 us)
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // a bounded wait gives up after 1 s
__device__ __forceinline__ unsigned saddr(const void *p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ unsigned long long globaltimer_ns() { return globaltimer_now(); }
__device__ __forceinline__ void mbar_init(uint64_t *b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
// one arrival that also announces `bytes` of asynchronous copies completing on the barrier
__device__ __forceinline__ void mbar_expect(uint64_t *b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
// test for the phase with the given parity; a waiting thread may be suspended (up to the hint, in
// nanoseconds) until the phase completes, so the wait costs no issue slots
__device__ __forceinline__ bool mbar_test(uint64_t *b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity), "r"(kWaitHintNs)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity. Returns false, without waiting, once *bad is set
// (another wait of the CTA gave up), and gives up itself (setting *bad) when the phase has not
// completed kWaitLimitNs after the wait began.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, unsigned parity, volatile int *bad) {
    if (*bad) return false;
    if (mbar_test(b, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (*bad) return false;
        if (mbar_test(b, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *bad = 1;
            return false;
        }
    }
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16) completing on barrier b
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *b) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(saddr(dst)),
                 "l"(src), "r"(bytes), "r"(saddr(b))
                 : "memory");
}

// Sum over the 16 lanes of a half warp (all 32 lanes must call).
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide sum with a fixed reduction order (deterministic). blockDim.x a multiple of 32, <= 1024.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    if (w == 0) {
        t = lane < nw ? red[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0) red[32] = t;
    }
    __syncthreads();
    return red[32];
}

// The segment partials a product launched with EPI_PART leaves: element (row m, column n) is the sum,
// in segment order, of part[((n/32 * maxseg + s) * 16 + m) * 32 + n % 32] over the nseg segments of
// quad q = n/128 (the CTAs whose unit ranges touch the quad's C chunks; the split of a grid of G CTAs
// over U = quads * C units gives CTA b the units [b*U/G, (b+1)*U/G)).
struct PartView {
    const float *part;
    int C, G, maxseg;
    long U;
};
__host__ __device__ __forceinline__ long cta_of(long u, long U, int G) { return ((u + 1) * G - 1) / U; }

// ---- row step arguments (row kernel, and products that finish their rows: EPI_ROWS) ------------------
struct RowArgs {
    int M, H;
    float *x;              // fp32 residual [M][H]
    const float *y;        // fp32 product [M][ldy] to add (nullable)
    int ldy;
    PartView yp;           // or the product as segment partials (yp.part non-null; takes precedence)
    float *y_out;          // the product's rows as fp32 [M][H] (nullable; for inspection)
    const uint16_t *w_post;   // RMSNorm weight applied to y before the add (nullable: plain add)
    float lambda;          // multiply x after the add (1 = none)
    float *tap;            // tap store base (nullable), row of position p at tap + p*ld_tap + tap_off
    int ld_tap, tap_off;
    const uint16_t *w_next;   // RMSNorm weight for the output (nullable: output = x)
    uint32_t *outf;        // output rows in operand format with H inputs (nullable)
    float *outs;           // their per-16 sums
    int out_row0;          // first output row
    float *out32;          // or output rows as fp32 [M][H] (nullable)
    float eps;
    const DevState *st;
    int pos_from_ctx;      // tap positions: 0 = st->n + m, 1 = st->draft_n + m
    int rows_from_ctx;     // 1: only rows < st->ctx_rows are live (the rest are written as zeros)
    Stamp ps;
};

struct QkArgs {
    int M, nq, nkv, hd;
    const float *qkv;      // fp32 [M][ldq] (q | k | v)
    int ldq;
    PartView qp;           // or the product as segment partials (qp.part non-null; takes precedence)
    float *qkv_out;        // the product's rows as fp32 [.][ldq] (nullable; for inspection)
    int row0;              // first row of qkv that belongs to this group of rows
    const uint16_t *q_norm, *k_norm;
    float eps;
    const float2 *rope;    // (cos, sin) table [max_pos][hd/2]
    const DevState *st;
    int pos_mode;          // 0: st->n + m, 1: st->n + m (draft block), 2: st->draft_n + m (draft context)
    int live_from_ctx;     // 1: only rows < st->ctx_rows are live
    float *q_out;          // fp32 [M][nq][hd] (nullable: no query)
    float *k_store, *v_store;      // [cap][nkv][hd] (nullable: no append)
    int cap;               // ring capacity (slot = pos % cap)
    Stamp ps;
};

// ---- GEMM interface ---------------------------------------------------------------------------------
enum WFmt { W_Q41 = 0, W_BF16 = 1 };
// EPI_PART: each CTA only writes its segment partial of every quad it touches (no fix-up); the
// consumer adds the segments (PartView).
// EPI_ROWS: as EPI_PART, then the last CTAs to finish perform the row step (RowArgs) of the rows.
// EPI_QK: as EPI_PART, then the last CTAs to finish perform the q/k steps (QkArgs) of the rows.
enum Epi { EPI_F32 = 0, EPI_GLU = 1, EPI_SILU_MUL = 2, EPI_ARGMAX = 3, EPI_PART = 4, EPI_ROWS = 5, EPI_QK = 6 };
enum ArgmaxDst { AM_VERIFY = 0, AM_DRAFT = 1, AM_OUT = 2 };

struct GemmArgs {
    const uint8_t *img;    // tile image
    int K, C, N;           // logical K, chunks of 64 along padded K, output columns
    int M;                 // rows (<= 16)
    const uint32_t *xf;    // activations, operand format (K inputs)
    const float *xs;       // their per-16 sums
    int x_row0;            // first activation row used
    int *err;              // products: sticky error bits (nullable), kErrWaitTimeout
    int skip_on_err;       // 1: a launch that finds *err set on entry issues no copies (the pass it
                           // belongs to has already failed) and its results are undefined
    int stall;             // test of the give-up path: the copy warp issues nothing, so every wait of
                           // the compute warps gives up (kErrWaitTimeout); 0 in normal use
    float *y;              // EPI_F32: fp32 output [M][ldy]
    int ldy;
    uint32_t *yf;          // EPI_GLU / EPI_SILU_MUL: output in operand format (N/2 or N inputs)
    float *ys;
    float *part;           // segment partials [N/32][maxseg][16][32]
    int maxseg;
    int *cnt;              // arrival counters [N/32] (zero between launches)
    const uint16_t *ext;   // EPI_SILU_MUL: bf16 multiplier [M][lde]
    int lde;
    // EPI_ARGMAX
    float *logits;         // optional fp32 [M][ldl] store of the raw products
    int ldl;
    float *am_val;         // per-CTA partial maxima [gridDim.x][M]
    int *am_idx;
    int *am_cnt;           // CTA arrival counter (zero between launches)
    DevState *st;
    int am_dst;            // AM_VERIFY: st->target[m] and st->accepted; AM_DRAFT: st->props[m];
                           // AM_OUT: am_out[m] (the standalone head)
    int *am_out;
    // EPI_ROWS / EPI_QK
    RowArgs row;           // the row step (row.yp: this launch's partials)
    QkArgs qk[2];          // the q/k steps (qk[i].qp: this launch's partials), nqk of them
    int nqk;
    int *row_cnt;          // [2] arrivals and finished workers (zero between launches)
    Stamp ps;              // profiling stamp (ps.prof == nullptr: none)
};

__device__ __forceinline__ float part_sum(const PartView &v, int m, int n) {
    const int grp = n >> 5, q = grp >> 2;
    const long qa = (long)q * v.C;
    const int nseg = int(cta_of(qa + v.C - 1, v.U, v.G) - cta_of(qa, v.U, v.G)) + 1;
    const float *p = v.part + ((size_t)grp * v.maxseg * kMaxRows + m) * 32 + (n & 31);
    float l[16];
#pragma unroll
    for (int s = 0; s < 16; ++s) l[s] = s < nseg ? __ldcg(p + (size_t)s * kMaxRows * 32) : 0.f;
    float y = 0.f;
#pragma unroll
    for (int s = 0; s < 16; ++s)
        if (s < nseg) y += l[s];
    for (int s = 16; s < nseg; ++s) y += __ldcg(p + (size_t)s * kMaxRows * 32);
    return y;
}

// launchers (gemm.cu)
int gemm_grid(int C, int N);
int gemm_maxseg(int C, int N);
size_t gemm_scratch_floats(int C, int N);
size_t gemm_part_floats(int C, int N);   // partials of an EPI_PART launch
cudaError_t launch_gemm(int fmt, int epi, const GemmArgs &a, cudaStream_t s);
int head_grid(int C, int M, int N);   // CTAs of a head launch (per-CTA maxima: head_grid * kMaxRows)
cudaError_t launch_act_pack(const float *x, int M, int K, uint32_t *f, float *sums, cudaStream_t s);
inline size_t act_words(int K) { return (size_t)kMaxRows * K; }          // fragment words of a 16-row buffer
inline size_t act_sums(int K) { return (size_t)(K / 16) * kMaxRows; }     // sum floats
cudaError_t launch_pack_q41(const uint8_t *src, int K, int N, uint8_t *img, cudaStream_t s);
cudaError_t launch_pack_bf16(const uint16_t *src, int K, int N, uint8_t *img, cudaStream_t s);
__host__ __device__ inline int padded_k(int K) { return (K + 63) / 64 * 64; }
inline size_t q41_image_bytes(int K, int N) { return size_t(N / 16) * (padded_k(K) / 64) * 640; }
inline size_t bf16_image_bytes(int K, int N) { return size_t(N / 16) * (padded_k(K) / 64) * 2048; }

// ---- row and attention interfaces (rows.cu) ------------------------------------------------------

struct EmbedArgs {
    int M, H;
    const uint16_t *emb;   // bf16 [vocab][H]
    float scale;
    const DevState *st;
    int use_draft;         // 0: tokens st->rows[m] (or tokens[m]); 1: draft block [st->last_tok, mask...]
    const int32_t *tokens; // row tokens [M] (nullable: st->rows)
    int mask_token;
    float *x;              // fp32 [M][H]
    const uint16_t *ple;   // bf16 [vocab][ple_w] (nullable)
    int ple_w;
    uint16_t *ple_out;     // bf16 [M][ple_w]
    Stamp ps;
};


struct AttnArgs {
    int M, nq, nkv, hd;
    const float *q;        // fp32 [M][nq][hd]
    const float *kA, *vA;      // positional store [capA][nkv][hd]
    int capA;
    const float *kB, *vB;      // block store [nB][nkv][hd] (nullable)
    int nB;
    int window;            // mode 0: keys p-window+1..p (0 = all of 0..p); mode 1: context window
    int mode;              // 0: target (causal, keys in A up to the row's own position)
                           // 1: draft (A keys max(0,n-window)..n-1 for every row, plus all B keys)
    const DevState *st;
    float scale;
    int *err;              // sticky error bits (nullable), kErrWaitTimeout
    int max_cluster;       // largest cluster size allowed (16, 8 or 4); the largest that fits is taken
    uint32_t *outf;        // [M][nq*hd] in operand format (M <= 16)
    float *outs;
    float *out32;          // or fp32 [M][nq*hd]; then M may exceed 16 (tiles of 16 rows, grid y)
    Stamp ps;
};

// The per-layer-embedding tail's two products in one launch (rows.cu, k_ple)
struct PleArgs {
    int M, H, P;
    const uint8_t *img_g;   // Q4_1 tile image of the gate, K = H, N = P
    const uint8_t *img_p;   // Q4_1 tile image of the projection, K = P, N = H
    const uint32_t *xf;     // the gate's input rows in operand format (H inputs, rows from 0)
    const float *xs;        // their per-16 sums
    const uint16_t *ext;    // the layer's per-layer-embedding rows: bf16, row m at ext + m * lde
    int lde;
    float *y;               // fp32 [M][H]: the projection's rows
    Stamp ps;
};
bool ple_fused_ok(int M, int H, int P);

struct SampleArgs {
    const float *logits;   // [M][V]
    int M, V, ld;
    int row0;              // the pass row of logits row 0 (its token is for position n + row0 + 1)
    DevState *st;
    int *cnt;
    Stamp ps;
};

cudaError_t launch_set_state(DevState *st, const SetStateArgs &a, cudaStream_t s);
cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t s);
cudaError_t launch_rows(const RowArgs &a, cudaStream_t s);
cudaError_t launch_qk(const QkArgs &a, cudaStream_t s);
cudaError_t launch_attn(const AttnArgs &a, cudaStream_t s);
cudaError_t attn_prepare(int hd);   // once per head dimension, outside stream capture
cudaError_t launch_sample(const SampleArgs &a, cudaStream_t s);
cudaError_t launch_rope_table(float2 *tab, int max_pos, int hd, double base, cudaStream_t s);
cudaError_t launch_cast_rows(const float *src, int ld_src, int M, int H, const uint16_t *w_norm, float eps,
                             uint32_t *dstf, float *dsts, int row0, const DevState *st, int live_from_ctx,
                             cudaStream_t s);
cudaError_t launch_copy_taps(const float *taps, int ld, const DevState *st, int M, uint32_t *dstf, cudaStream_t s);
cudaError_t launch_plant(DevState *st, const int32_t *table, int count, cudaStream_t s);
cudaError_t launch_ple(const PleArgs &a, cudaStream_t s);
// fp32 rows of a long pass: out[m][j] = silu(y[m][j]) * y[m][F + j] (gate | up halves of a product row)
cudaError_t launch_glu32(const float *y, int M, int F, float *out, cudaStream_t s);
// out[m][j] = silu(y[m][j]) * e[m * lde + j] (bf16 e)
cudaError_t launch_silu_mul32(const float *y, int M, int P, const uint16_t *e, int lde, float *out, cudaStream_t s);
// the Q4_1 product of many fp32 rows on the tcgen05 tensor cores (tcgemm.cu); scratch 1024-byte aligned
size_t tc_gemm_scratch_bytes(int K, int N, int M);
cudaError_t launch_tc_gemm(const uint8_t *img, int K, int N, const float *x, int M, float *y, void *scratch,
                           int *err, cudaStream_t s);

// Launch with programmatic stream serialization (kernels begin with pdl_wait()).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}


}  // namespace dfl
