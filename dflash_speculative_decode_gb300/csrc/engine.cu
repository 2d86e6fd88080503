// engine.cu -- host engine behind the C ABI (include/dfl.h): arena layout, tensor packing, the
// sequence of kernels of a verify / prefill chunk / draft block, and the index arithmetic of commit,
// snapshot and restore.
//
// State (1bit engine PR "npu forward: Gemma4 verifies a draft in one batched pass; KV row width per
// layer", "What changes" item 1): one KV plane per layer that holds its own, counted at that layer's
// width (2 * kv_heads * head_dim floats per position); a KV-shared layer holds none and reads its
// owner's; positions held are counted over owner planes. Sliding planes are rings of W + R_max - 1
// slots (a verify writes up to R_max rows before knowing how many survive, and the oldest key a later
// row needs is W - 1 behind it), full planes are linear. commit_verify_rows only moves the position
// counter: rows past it are overwritten by the next pass.
#include <algorithm>
#include <cctype>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "dfl.h"
#include "rowstep.cuh"

// A named NVTX range around each pass-level call, so that a profiler's timeline (and ncu's --nvtx-include
// filter) can tell prefill, draft and verify passes apart. The NVTX v3 header needs no library; without a
// tool attached the calls do nothing. A toolkit without the header builds the ranges as no-ops.
#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#else
struct NvtxRange {
    explicit NvtxRange(const char *) {}
};
#endif

namespace dfl {
size_t attn_smem(int M, int hd);
}  // namespace dfl

using namespace dfl;

namespace {

struct QMat {
    uint8_t *img = nullptr;
    int K = 0, N = 0, C = 0, maxseg = 1;
    bool q41 = true;
    bool loaded = false;
};
// a 16-row activation buffer in the products' operand format
struct Act {
    uint32_t *f = nullptr;
    float *s = nullptr;
};
struct Vec {
    uint16_t *p = nullptr;
    size_t n = 0;
    bool loaded = false;
};
struct TLayer {
    int type = 0, owner = 0, nkv = 0, ffn = 0, cap = 0;
    QMat qkv, o, gu, d, pg, pp;
    Vec attn_norm, q_norm, k_norm, post_attn_norm, pre_ffn_norm, post_ffn_norm, ple_norm, lam;
    float lambda = 1.f;
    float *K = nullptr, *V = nullptr;
};
struct DLayer {
    QMat qkv, o, gu, d;
    Vec attn_norm, q_norm, k_norm, ffn_norm;
    float *K = nullptr, *V = nullptr;
};

struct Arena {
    uint8_t *base = nullptr;
    size_t off = 0;
    template <typename T>
    T *take(size_t count) {
        off = (off + 255) / 256 * 256;
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

uint64_t fnv1a(const void *p, size_t n) {
    const uint8_t *b = static_cast<const uint8_t *>(p);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < n; ++i) h = (h ^ b[i]) * 1099511628211ull;
    return h;
}

constexpr uint32_t kSnapMagic = 0x53464C44u;   // "DLFS"

struct SnapHeader {
    uint32_t magic, version;
    uint64_t cfg_hash;
    int32_t n, draft_n;
    uint64_t bytes;
    uint8_t pad[224];
};
static_assert(sizeof(SnapHeader) == 256, "header size");

}  // namespace

constexpr int kProfClasses = 6;

struct dfl_ctx {
    dfl_config cfg{};
    cudaStream_t stream = nullptr;
    // weights
    Vec emb, final_norm, ple_table, d_hidden_norm, d_final_norm;
    QMat head, fc;
    std::vector<TLayer> tl;
    std::vector<DLayer> dl;
    float2 *rope_s = nullptr, *rope_f = nullptr, *rope_d = nullptr;
    int rope_rows = 0;
    // state
    DevState *st = nullptr;
    float *taps = nullptr;
    int TH = 0, cap_sliding = 0, cap_draft = 0, ctx_fuse = 0;
    // workspace
    float *x = nullptr, *x_d = nullptr, *y = nullptr, *y_fc = nullptr, *qkv = nullptr, *q = nullptr;
    float *part = nullptr, *logits = nullptr, *dlogits = nullptr, *am_val = nullptr;
    Act h, hcat, hb, o, a, z, tapbuf;
    float *kB = nullptr, *vB = nullptr;
    uint16_t *ple_rows = nullptr;
    int *cnt = nullptr, *am_idx = nullptr, *am_cnt = nullptr, *smp_cnt = nullptr, *row_cnt = nullptr;
    int *counters_begin = nullptr;
    size_t counters_bytes = 0;
    int nq_max = 0, qkv_max = 0;
    // a long prefill pass: its tokens, residual rows, two fp32 row buffers, PLE rows, product scratch
    int32_t *pf_tok = nullptr;
    float *pf_x = nullptr, *pf_a = nullptr, *pf_b = nullptr;
    uint16_t *pf_ple = nullptr;
    uint8_t *pf_scratch = nullptr;
    // host mirror of the state
    int n = 0, draft_n = 0, pending = 0, last_accepted = -1, draft_at = -1;
    int draft_n_ok = 0;       // draft_n as of the last call that read the device state without an error
    int32_t last_target[kMaxRows] = {};   // the target's tokens of the last verify
    bool test_stall = false;  // test of the give-up path: the products of the next passes issue no copies
    bool fuse_steps = false;  // the row and q/k steps run on the products' last CTAs (DFL_OPT_FUSE_STEPS)
    bool ple_split = false;   // the PLE gate and projection as two products (DFL_OPT_PLE_SPLIT)
    bool draft_only = false, keep_logits = false, have_logits = false, have_dlogits = false;
    // a failed prefill may have overwritten ring slots (sliding planes, the draft context) that the
    // positions held still need: passes and snapshots are refused until a restore
    bool needs_restore = false;
    int last_k = 0;
    int stop_layer = -1;   // debug: a target pass runs layers 0..stop_layer only (no head)
    int attn_cluster = 16; // largest attention cluster size allowed: 16, 8 or 4
    long long launches = 0;                       // kernels this context has launched
    bool profile = false;                         // stamp the instrumented launches of each pass
    unsigned long long *prof = nullptr;           // device stamps [2][kProfSlots] (workspace)
    int prof_next = 0;                            // next slot of the pass being built
    struct Rec { int cls; double bytes; int slot; };
    std::vector<Rec> recs;                        // profiled launches of the pass being built
    std::vector<unsigned long long> prof_host;
    double prof_ms[kProfClasses] = {}, prof_bytes[kProfClasses] = {};
    long long prof_n[kProfClasses] = {};
    // captured passes
    bool use_graphs = true, capturing = false;
    cudaStream_t cap_stream = nullptr;
    struct Graph {
        cudaGraphExec_t exec = nullptr;
        std::vector<Rec> recs;                    // profiled launches inside the graph
        long long launches = 0;                   // kernels per replay
    };
    std::map<uint64_t, Graph> graphs;
    std::string err;
};

namespace {

int fail(dfl_ctx *c, int code, const std::string &msg) {
    if (c) c->err = msg;
    return code;
}

#define DFL_CK(call)                                                                          \
    do {                                                                                      \
        cudaError_t e_ = (call);                                                              \
        if (e_ != cudaSuccess) return fail(c, DFL_E_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
    } while (0)

// a kernel launch (not stamped; its time is not in any class)
#define DFL_LAUNCH_C(cls, call)                                                               \
    do {                                                                                      \
        c->launches += 1;                                                                     \
        DFL_CK(call);                                                                         \
    } while (0)
#define DFL_LAUNCH(call) DFL_LAUNCH_C(5, call)
// a stamped kernel launch of profiling class `cls`: the argument struct gets its profiling slot
#define DFL_LAUNCH_S(cls, args, launcher)                                                     \
    do {                                                                                      \
        (args).ps = stamp(c, cls, 0.0);                                                       \
        DFL_LAUNCH_C(cls, launcher(args, c->stream));                                         \
    } while (0)

std::string validate(const dfl_config *g) {
    auto bad = [](const char *f) { return std::string("configuration: ") + f; };
    if (g->n_layers < 1 || g->n_layers > DFL_MAX_LAYERS) return bad("n_layers out of range 1..64");
    if (g->hidden < 128 || g->hidden % 128 || g->hidden > 8192) return bad("hidden must be a multiple of 128, <= 8192");
    if (g->vocab < 16 || g->vocab % 16) return bad("vocab must be a multiple of 16");
    if (g->head_dim != 64 && g->head_dim != 128 && g->head_dim != 256) return bad("head_dim must be 64, 128 or 256");
    if (g->n_heads < 1 || (g->n_heads * g->head_dim) % 64) return bad("n_heads * head_dim must be a multiple of 64");
    if (g->window < 1) return bad("window must be >= 1");
    if (g->ple_dim < 0 || g->ple_dim % 32) return bad("ple_dim must be a multiple of 32");
    for (int l = 0; l < g->n_layers; ++l) {
        const int o = g->kv_owner[l], t = g->layer_type[l], kv = g->kv_heads[l];
        if (t != DFL_SLIDING && t != DFL_FULL) return bad("layer_type must be 0 or 1");
        if (kv < 1 || g->n_heads % kv) return bad("kv_heads must divide n_heads");
        if (o < 0 || o > l) return bad("kv_owner must be an earlier layer or the layer itself");
        if (o != l && (g->kv_owner[o] != o || g->layer_type[o] != t || g->kv_heads[o] != kv))
            return bad("a KV-shared layer's owner must hold its own plane, of the same type and kv_heads");
        if (g->ffn[l] < 64 || g->ffn[l] % 64) return bad("ffn must be a multiple of 64");
        if (((g->n_heads + 2 * kv) * g->head_dim) % 32) return bad("q|k|v width must be a multiple of 32");
    }
    if (g->d_layers < 1 || g->d_layers > DFL_MAX_LAYERS) return bad("d_layers out of range");
    if (g->d_head_dim != 64 && g->d_head_dim != 128 && g->d_head_dim != 256) return bad("d_head_dim must be 64, 128 or 256");
    if (g->d_heads < 1 || g->d_kv_heads < 1 || g->d_heads % g->d_kv_heads) return bad("d_kv_heads must divide d_heads");
    if ((g->d_heads * g->d_head_dim) % 64) return bad("d_heads * d_head_dim must be a multiple of 64");
    if (g->d_ffn < 64 || g->d_ffn % 64) return bad("d_ffn must be a multiple of 64");
    if (g->d_window < 0) return bad("d_window must be >= 0");
    if (g->block < 2 || g->block > DFL_MAX_ROWS) return bad("block must be 2..16");
    if (g->n_taps < 1 || g->n_taps > DFL_MAX_TAPS) return bad("n_taps must be 1..8");
    for (int i = 0; i < g->n_taps; ++i) {
        if (g->taps[i] < 0 || g->taps[i] >= g->n_layers) return bad("tap layer out of range");
        if (i && g->taps[i] <= g->taps[i - 1]) return bad("taps must be ascending");
    }
    if (g->mask_token < 0 || g->mask_token >= g->vocab) return bad("mask_token out of range");
    if (g->max_ctx < 1 || g->max_ctx > (1 << 20)) return bad("max_ctx out of range");
    if (!(g->eps > 0.f) || !(g->d_eps > 0.f)) return bad("eps must be > 0");
    if (g->prefill_rows != 0 && (g->prefill_rows < 128 || g->prefill_rows > 8192 || g->prefill_rows % 16))
        return bad("prefill_rows must be 0 or 128..8192, a multiple of 16");
    return {};
}

QMat qmat(int K, int N, bool q41) {
    QMat m;
    m.K = K;
    m.N = N;
    m.C = padded_k(K) / 64;
    m.maxseg = gemm_maxseg(m.C, N);
    m.q41 = q41;
    return m;
}

// Lay out every buffer. With null bases only the sizes are computed.
void plan(dfl_ctx *c, Arena &W, Arena &S, Arena &X) {
    const dfl_config &g = c->cfg;
    const int H = g.hidden, V = g.vocab, NL = g.n_layers, hd = g.head_dim, nq = g.n_heads, P = g.ple_dim;
    const int R = kMaxRows;
    c->TH = g.n_taps * H;
    const int PF = g.prefill_rows;
    // a sliding ring holds the window of the first row of a pass plus the pass's own rows
    c->cap_sliding = g.window + std::max(R, PF) - 1;
    c->cap_draft = g.d_window > 0 ? g.d_window : g.max_ctx + R;
    c->ctx_fuse = R - g.block;
    c->rope_rows = g.max_ctx + 2 * R;

    size_t part_floats = 0;
    int cnt_n = 1;
    auto qm = [&](QMat &m, int K, int N, bool q41) {
        m = qmat(K, N, q41);
        m.img = W.take<uint8_t>(q41 ? q41_image_bytes(K, N) : bf16_image_bytes(K, N));
        part_floats = std::max(part_floats, gemm_part_floats(m.C, N));
        cnt_n = std::max(cnt_n, N / 32);
    };
    auto vec = [&](Vec &v, size_t n) {
        v.n = n;
        v.p = W.take<uint16_t>(n);
    };
    vec(c->emb, (size_t)V * H);
    qm(c->head, H, V, false);
    vec(c->final_norm, H);
    if (P) vec(c->ple_table, (size_t)V * NL * P);
    c->tl.assign(NL, TLayer());
    c->qkv_max = 0;
    int ffn_max = g.d_ffn;
    for (int l = 0; l < NL; ++l) {
        TLayer &L = c->tl[l];
        L.type = g.layer_type[l];
        L.owner = g.kv_owner[l];
        L.nkv = g.kv_heads[l];
        L.ffn = g.ffn[l];
        ffn_max = std::max(ffn_max, L.ffn);
        const bool own = L.owner == l;
        const int nqkv = (nq + (own ? 2 * L.nkv : 0)) * hd;
        c->qkv_max = std::max(c->qkv_max, nqkv);
        vec(L.attn_norm, H);
        vec(L.q_norm, hd);
        if (own) vec(L.k_norm, hd);
        vec(L.post_attn_norm, H);
        vec(L.pre_ffn_norm, H);
        vec(L.post_ffn_norm, H);
        qm(L.qkv, H, nqkv, true);
        qm(L.o, nq * hd, H, true);
        qm(L.gu, H, 2 * L.ffn, true);
        qm(L.d, L.ffn, H, true);
        if (P) {
            vec(L.ple_norm, H);
            vec(L.lam, 1);
            qm(L.pg, H, P, true);
            qm(L.pp, P, H, true);
        }
    }
    const int dq = g.d_heads, dkv = g.d_kv_heads, dhd = g.d_head_dim;
    qm(c->fc, c->TH, H, false);
    vec(c->d_hidden_norm, H);
    vec(c->d_final_norm, H);
    c->dl.assign(g.d_layers, DLayer());
    for (int l = 0; l < g.d_layers; ++l) {
        DLayer &D = c->dl[l];
        vec(D.attn_norm, H);
        vec(D.q_norm, dhd);
        vec(D.k_norm, dhd);
        vec(D.ffn_norm, H);
        qm(D.qkv, H, (dq + 2 * dkv) * dhd, true);
        qm(D.o, dq * dhd, H, true);
        qm(D.gu, H, 2 * g.d_ffn, true);
        qm(D.d, g.d_ffn, H, true);
    }
    c->qkv_max = std::max(c->qkv_max, (dq + 2 * dkv) * dhd);
    c->rope_s = W.take<float2>((size_t)c->rope_rows * (hd / 2));
    c->rope_f = W.take<float2>((size_t)c->rope_rows * (hd / 2));
    c->rope_d = W.take<float2>((size_t)c->rope_rows * (dhd / 2));

    // state
    c->st = S.take<DevState>(1);
    for (int l = 0; l < NL; ++l) {
        TLayer &L = c->tl[l];
        if (L.owner != l) continue;
        L.cap = L.type == DFL_SLIDING ? c->cap_sliding : g.max_ctx + R;
        L.K = S.take<float>((size_t)L.cap * L.nkv * hd);
        L.V = S.take<float>((size_t)L.cap * L.nkv * hd);
    }
    for (int l = 0; l < g.d_layers; ++l) {
        c->dl[l].K = S.take<float>((size_t)c->cap_draft * dkv * dhd);
        c->dl[l].V = S.take<float>((size_t)c->cap_draft * dkv * dhd);
    }
    c->taps = S.take<float>((size_t)(g.max_ctx + 2 * R) * c->TH);

    // workspace
    c->nq_max = std::max(nq, dq);
    const int hd_max = std::max(hd, dhd);
    const int att_max = std::max(nq * hd, dq * dhd);
    c->x = X.take<float>((size_t)R * H);
    c->x_d = X.take<float>((size_t)R * H);
    c->y = X.take<float>((size_t)R * H);
    c->y_fc = X.take<float>((size_t)R * H);
    c->qkv = X.take<float>((size_t)R * c->qkv_max);
    c->q = X.take<float>((size_t)R * att_max);
    auto act = [&](Act &A, int K) {
        A.f = X.take<uint32_t>(act_words(K));
        A.s = X.take<float>(act_sums(K));
    };
    act(c->h, H);
    act(c->hcat, H);
    act(c->hb, H);
    act(c->o, att_max);
    act(c->a, ffn_max);
    act(c->z, std::max(P, 32));
    c->ple_rows = X.take<uint16_t>((size_t)R * std::max(NL * P, 32));
    act(c->tapbuf, c->TH);
    c->kB = X.take<float>((size_t)R * dkv * dhd);
    c->vB = X.take<float>((size_t)R * dkv * dhd);
    c->part = X.take<float>(std::max<size_t>(part_floats, 1));
    c->am_val = X.take<float>((size_t)152 * 4 * kMaxRows);
    c->am_idx = X.take<int>((size_t)152 * 4 * kMaxRows);
    c->prof = X.take<unsigned long long>(2 * (size_t)kProfSlots);
    c->logits = X.take<float>((size_t)R * V);
    c->dlogits = X.take<float>((size_t)R * V);
    // buffers of a long prefill pass (rows past 16; products on the tcgen05 tensor cores)
    if (PF) {
        int wmax = std::max(std::max(H, nq * hd), std::max(c->qkv_max, 2 * ffn_max));
        wmax = std::max(wmax, P);
        c->pf_tok = X.take<int32_t>(PF);
        c->pf_x = X.take<float>((size_t)PF * H);
        c->pf_a = X.take<float>((size_t)PF * wmax);
        c->pf_b = X.take<float>((size_t)PF * wmax);
        c->pf_ple = X.take<uint16_t>((size_t)PF * std::max(NL * P, 32));
        size_t sb = 0;
        for (int l = 0; l < NL; ++l) {
            const TLayer &L = c->tl[l];
            for (const QMat *m : {&L.qkv, &L.o, &L.gu, &L.d})
                sb = std::max(sb, tc_gemm_scratch_bytes(m->K, m->N, PF));
            if (P) {
                sb = std::max(sb, tc_gemm_scratch_bytes(L.pg.K, L.pg.N, PF));
                sb = std::max(sb, tc_gemm_scratch_bytes(L.pp.K, L.pp.N, PF));
            }
        }
        uint8_t *raw = X.take<uint8_t>(sb + 1024);
        c->pf_scratch = raw ? reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023))
                            : nullptr;
    }
    // counters that must read zero between launches, contiguous so one memset clears them
    X.off = (X.off + 255) / 256 * 256;
    const size_t cbeg = X.off;
    c->cnt = X.take<int>(cnt_n);
    c->am_cnt = X.take<int>(1);
    c->smp_cnt = X.take<int>(1);
    c->row_cnt = X.take<int>(2);
    c->counters_begin = c->cnt;
    c->counters_bytes = X.off - cbeg;
}

bool is_tap(const dfl_config &g, int l, int *ti) {
    for (int i = 0; i < g.n_taps; ++i)
        if (g.taps[i] == l) {
            *ti = i;
            return true;
        }
    return false;
}

// ---- one product -----------------------------------------------------------------------------------
// profiled launch classes: 0 = Q4_1 products, 1 = bf16 products (fc), 2 = head, 3 = attention,
// 4 = q/k norm + rotation + KV store, 5 = row kernels (residual, norms, taps), embedding, sampling.
// The small state and copy kernels are not stamped.
Stamp stamp(dfl_ctx *c, int cls, double bytes) {
    if (!c->profile || c->prof_next >= kProfSlots) return Stamp{nullptr, 0};
    const int slot = c->prof_next++;
    c->recs.push_back({cls, bytes, slot});
    return Stamp{c->prof, slot};
}

// y = x . W for M rows; EPI_F32 writes fp32 rows to y, EPI_GLU / EPI_SILU_MUL write `out` in operand format
cudaError_t gemm(dfl_ctx *c, const QMat &W, const Act &x, int row0, int M, int epi, float *y, int ldy,
                 const Act *out = nullptr, const uint16_t *ext = nullptr, int lde = 0, const RowArgs *row = nullptr,
                 const QkArgs *qk0 = nullptr, const QkArgs *qk1 = nullptr) {
    GemmArgs a{};
    if (row) a.row = *row;
    if (qk0) a.qk[0] = *qk0, a.nqk = 1;
    if (qk1) a.qk[1] = *qk1, a.nqk = 2;
    a.row_cnt = c->row_cnt;
    a.img = W.img;
    a.K = W.K;
    a.C = W.C;
    a.N = W.N;
    a.M = M;
    a.xf = x.f;
    a.xs = x.s;
    a.x_row0 = row0;
    a.y = y;
    a.ldy = ldy;
    a.yf = out ? out->f : nullptr;
    a.ys = out ? out->s : nullptr;
    a.part = c->part;
    a.maxseg = W.maxseg;
    a.cnt = c->cnt;
    a.ext = ext;
    a.lde = lde;
    a.err = &c->st->err;
    a.skip_on_err = 1;
    a.stall = c->test_stall ? 1 : 0;
    a.ps = stamp(c, W.q41 ? 0 : 1, (W.q41 ? 0.625 : 2.0) * W.K * (double)W.N + 4.0 * M * W.K + 4.0 * M * W.N);
    c->launches += 1;
    return launch_gemm(W.q41 ? W_Q41 : W_BF16, epi, a, c->stream);
}

// the segment partials an EPI_PART product of W leaves in the context's partial buffer
PartView part_view(const dfl_ctx *c, const QMat &W) {
    PartView v{};
    v.part = c->part;
    v.C = W.C;
    v.G = gemm_grid(W.C, W.N);
    v.maxseg = W.maxseg;
    v.U = (long)((W.N / 32 + 3) / 4) * W.C;
    return v;
}

// a product whose last CTAs also perform the row step r of its rows (r.yp: this product's partials);
// rows wider than the product's row step takes run the row kernel after the product instead
cudaError_t gemm_rows(dfl_ctx *c, const QMat &W, const Act &x, int M, RowArgs r) {
    r.yp = part_view(c, W);
    if (c->fuse_steps && r.H <= kProductRowCols)
        return gemm(c, W, x, 0, M, EPI_ROWS, nullptr, 0, nullptr, nullptr, 0, &r);
    cudaError_t e = gemm(c, W, x, 0, M, EPI_PART, nullptr, 0);
    if (e != cudaSuccess) return e;
    r.ps = stamp(c, 5, 0.0);
    c->launches += 1;
    return launch_rows(r, c->stream);
}

// a q|k|v product whose last CTAs also perform the q/k steps q0 (and q1) of its rows
cudaError_t gemm_qk(dfl_ctx *c, const QMat &W, const Act &x, int M, QkArgs q0, const QkArgs *q1 = nullptr) {
    q0.qp = part_view(c, W);
    QkArgs b{};
    if (q1) {
        b = *q1;
        b.qp = q0.qp;
    }
    if (c->fuse_steps)
        return gemm(c, W, x, 0, M, EPI_QK, nullptr, 0, nullptr, nullptr, 0, nullptr, &q0, q1 ? &b : nullptr);
    cudaError_t e = gemm(c, W, x, 0, M, EPI_PART, nullptr, 0);
    if (e != cudaSuccess) return e;
    for (QkArgs *q : {&q0, q1 ? &b : nullptr}) {
        if (!q) continue;
        q->ps = stamp(c, 4, 0.0);
        c->launches += 1;
        e = launch_qk(*q, c->stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t head(dfl_ctx *c, const Act &x, int row0, int M, float *logits, int dst) {
    GemmArgs a{};
    a.img = c->head.img;
    a.K = c->head.K;
    a.C = c->head.C;
    a.N = c->head.N;
    a.M = M;
    a.xf = x.f;
    a.xs = x.s;
    a.x_row0 = row0;
    a.logits = logits;
    a.ldl = c->cfg.vocab;
    a.am_val = c->am_val;
    a.am_idx = c->am_idx;
    a.am_cnt = c->am_cnt;
    a.st = c->st;
    a.am_dst = dst;
    a.ps = stamp(c, 2, 2.0 * a.K * (double)a.N + 4.0 * M * a.K + (logits ? 4.0 * M * a.N : 0.0));
    c->launches += 1;
    return launch_gemm(W_BF16, EPI_ARGMAX, a, c->stream);
}

// Fold the stamps of one profiled pass (its records `recs`) into the totals (synchronises).
cudaError_t harvest(dfl_ctx *c, const std::vector<dfl_ctx::Rec> &recs) {
    if (recs.empty()) return cudaSuccess;
    c->prof_host.resize(2 * kProfSlots);
    cudaError_t e = cudaMemcpyAsync(c->prof_host.data(), c->prof, 2 * kProfSlots * sizeof(unsigned long long),
                                    cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return e;
    for (const auto &r : recs) {
        const unsigned long long t0 = c->prof_host[r.slot], t1 = c->prof_host[kProfSlots + r.slot];
        if (t1 < t0) continue;   // the launch had no CTA (nothing to do)
        c->prof_ms[r.cls] += (t1 - t0) * 1e-6;
        c->prof_bytes[r.cls] += r.bytes;
        c->prof_n[r.cls] += 1;
    }
    return cudaSuccess;
}

// reset the stamps before a profiled pass: ready times to the maximum, done times to zero
cudaError_t prof_reset(dfl_ctx *c) {
    cudaError_t e = cudaMemsetAsync(c->prof, 0xFF, kProfSlots * sizeof(unsigned long long), c->stream);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(c->prof + kProfSlots, 0, kProfSlots * sizeof(unsigned long long), c->stream);
}

// Run a pass body either directly or as a CUDA graph captured once per key (on a private stream,
// replayed on the context's stream). The body must only enqueue kernels. A profiled pass is followed
// by a synchronising read of its stamps.
int run_graph(dfl_ctx *c, uint64_t key, const std::function<int()> &body) {
    c->prof_next = 0;
    c->recs.clear();
    if (!c->use_graphs) {
        if (c->profile) DFL_CK(prof_reset(c));
        const int rc = body();
        if (rc) return rc;
        if (c->profile) DFL_CK(harvest(c, c->recs));
        c->recs.clear();
        return DFL_OK;
    }
    key = (key * 2 + (c->profile ? 1 : 0)) * 2 + (c->test_stall ? 1 : 0);
    auto it = c->graphs.find(key);
    if (it == c->graphs.end()) {
        if (!c->cap_stream) DFL_CK(cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking));
        cudaStream_t user = c->stream;
        c->stream = c->cap_stream;
        c->capturing = true;
        const long long l0 = c->launches;
        cudaError_t e = cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal);
        int rc = e == cudaSuccess ? body() : DFL_E_CUDA;
        cudaGraph_t g = nullptr;
        cudaError_t e2 = cudaStreamEndCapture(c->cap_stream, &g);
        c->stream = user;
        c->capturing = false;
        if (e != cudaSuccess) return fail(c, DFL_E_CUDA, std::string("cudaStreamBeginCapture: ") + cudaGetErrorString(e));
        if (rc) {
            if (g) cudaGraphDestroy(g);
            return rc;
        }
        if (e2 != cudaSuccess) return fail(c, DFL_E_CUDA, std::string("cudaStreamEndCapture: ") + cudaGetErrorString(e2));
        dfl_ctx::Graph G;
        e = cudaGraphInstantiate(&G.exec, g, 0);
        cudaGraphDestroy(g);
        if (e != cudaSuccess) return fail(c, DFL_E_CUDA, std::string("cudaGraphInstantiate: ") + cudaGetErrorString(e));
        G.launches = c->launches - l0;
        c->launches = l0;
        G.recs = c->recs;
        c->recs.clear();
        it = c->graphs.emplace(key, G).first;
    }
    dfl_ctx::Graph &G = it->second;
    if (c->profile) DFL_CK(prof_reset(c));
    DFL_CK(cudaGraphLaunch(G.exec, c->stream));
    c->launches += G.launches;
    if (c->profile) DFL_CK(harvest(c, G.recs));
    return DFL_OK;
}

RowArgs rows(dfl_ctx *c, int M, float *x) {
    RowArgs r{};
    r.M = M;
    r.H = c->cfg.hidden;
    r.x = x;
    r.lambda = 1.f;
    r.eps = c->cfg.eps;
    r.st = c->st;
    return r;
}

int set_state(dfl_ctx *c, int k, const int32_t *rows_in, bool draft_rows, int ctx_rows, int last_tok,
              const dfl_sampling *s) {
    SetStateArgs a{};
    a.n = c->n;
    a.k = k;
    a.draft_n = c->draft_n;
    a.ctx_rows = ctx_rows;
    a.use_draft_rows = draft_rows ? 1 : 0;
    a.last_tok = last_tok;
    a.sampled = (s && s->temperature > 0.f) ? 1 : 0;
    a.temperature = a.sampled ? s->temperature : 1.f;
    a.seed = s ? s->seed : 0;
    for (int i = 0; i < kMaxRows; ++i) a.rows[i] = (rows_in && i < k) ? rows_in[i] : 0;
    DFL_LAUNCH(launch_set_state(c->st, a, c->stream));
    return DFL_OK;
}

// ---- target pass: k rows at positions n..n+k-1 ---------------------------------------------------------
// head_last: the head (and sampling) for the last row only (a prefill chunk needs only its last token)
int target_body(dfl_ctx *c, int k, bool do_head, bool sampled, bool head_last = false) {
    const dfl_config &g = c->cfg;
    const int H = g.hidden, NL = g.n_layers, hd = g.head_dim, nq = g.n_heads, P = g.ple_dim;
    EmbedArgs ea{};
    ea.M = k;
    ea.H = H;
    ea.emb = c->emb.p;
    ea.scale = g.emb_scale;
    ea.st = c->st;
    ea.x = c->x;
    ea.ple = P ? c->ple_table.p : nullptr;
    ea.ple_w = NL * P;
    ea.ple_out = c->ple_rows;
    DFL_LAUNCH_S(5, ea, launch_embed);
    RowArgs r0 = rows(c, k, c->x);
    r0.w_next = c->tl[0].attn_norm.p;
    r0.outf = c->h.f;
    r0.outs = c->h.s;
    DFL_LAUNCH_S(5, r0, launch_rows);
    const int last_layer = (c->stop_layer >= 0 && c->stop_layer < NL) ? c->stop_layer : NL - 1;
    if (last_layer < NL - 1) do_head = false;
    for (int l = 0; l <= last_layer; ++l) {
        TLayer &L = c->tl[l];
        TLayer &O = c->tl[L.owner];
        const bool own = L.owner == l;
        const int nqkv = L.qkv.N;
        QkArgs qa{};
        qa.M = k;
        qa.nq = nq;
        qa.nkv = L.nkv;
        qa.hd = hd;
        qa.qp = part_view(c, L.qkv);
        qa.qkv_out = c->qkv;
        qa.ldq = nqkv;
        qa.q_norm = L.q_norm.p;
        qa.k_norm = own ? L.k_norm.p : nullptr;
        qa.eps = g.eps;
        qa.rope = L.type == DFL_SLIDING ? c->rope_s : c->rope_f;
        qa.st = c->st;
        qa.q_out = c->q;
        qa.k_store = own ? L.K : nullptr;
        qa.v_store = own ? L.V : nullptr;
        qa.cap = L.cap;
        DFL_CK(gemm_qk(c, L.qkv, c->h, k, qa));   // its last CTAs norm, rotate and store q, k, v
        AttnArgs aa{};
        aa.M = k;
        aa.nq = nq;
        aa.nkv = L.nkv;
        aa.hd = hd;
        aa.q = c->q;
        aa.kA = O.K;
        aa.vA = O.V;
        aa.capA = O.cap;
        aa.window = L.type == DFL_SLIDING ? g.window : 0;
        aa.mode = 0;
        aa.st = c->st;
        aa.scale = 1.0f / sqrtf((float)hd);
        aa.err = &c->st->err;
        aa.max_cluster = c->attn_cluster;
        aa.outf = c->o.f;
        aa.outs = c->o.s;
        DFL_LAUNCH_S(3, aa, launch_attn);
        // each of the row steps below runs in the last CTAs of the product before it
        RowArgs r1 = rows(c, k, c->x);
        r1.y_out = c->y;
        r1.w_post = L.post_attn_norm.p;
        r1.w_next = L.pre_ffn_norm.p;
        r1.outf = c->h.f;
        r1.outs = c->h.s;
        DFL_CK(gemm_rows(c, L.o, c->o, k, r1));
        DFL_CK(gemm(c, L.gu, c->h, 0, k, EPI_GLU, nullptr, 0, &c->a));
        const uint16_t *next = l + 1 < NL ? c->tl[l + 1].attn_norm.p : c->final_norm.p;
        int ti = 0;
        const bool tap = is_tap(g, l, &ti);
        RowArgs r2 = rows(c, k, c->x);
        r2.y_out = c->y;
        r2.w_post = L.post_ffn_norm.p;
        r2.outf = c->h.f;
        r2.outs = c->h.s;
        const QMat *last = &L.d;
        bool ple_one = false;   // the PLE gate and projection in one launch, its rows in c->y
        if (P) {
            DFL_CK(gemm_rows(c, L.d, c->a, k, r2));   // out = x: the gate's input
            ple_one = !c->ple_split && ple_fused_ok(k, H, P);
            if (ple_one) {
                PleArgs pa{};
                pa.M = k;
                pa.H = H;
                pa.P = P;
                pa.img_g = L.pg.img;
                pa.img_p = L.pp.img;
                pa.xf = c->h.f;
                pa.xs = c->h.s;
                pa.ext = c->ple_rows + (size_t)l * P;
                pa.lde = NL * P;
                pa.y = c->y;
                pa.ps = stamp(c, 0, 2 * 0.625 * H * (double)P + 8.0 * k * H);
                DFL_LAUNCH_C(0, launch_ple(pa, c->stream));
            } else {
                DFL_CK(gemm(c, L.pg, c->h, 0, k, EPI_SILU_MUL, nullptr, 0, &c->z, c->ple_rows + (size_t)l * P, NL * P));
            }
            r2 = rows(c, k, c->x);
            r2.y_out = ple_one ? nullptr : c->y;
            r2.w_post = L.ple_norm.p;
            r2.lambda = L.lambda;
            r2.outf = c->h.f;
            r2.outs = c->h.s;
            last = &L.pp;
        }
        r2.w_next = next;
        if (tap) {
            r2.tap = c->taps;
            r2.ld_tap = c->TH;
            r2.tap_off = ti * H;
        }
        if (ple_one) {
            r2.y = c->y;   // the projection's rows, written by the PLE launch
            r2.ldy = H;
            DFL_LAUNCH_S(5, r2, launch_rows);
        } else {
            DFL_CK(gemm_rows(c, *last, P ? c->z : c->a, k, r2));
        }
    }
    if (do_head) {
        float *lg = (c->keep_logits || sampled) ? c->logits : nullptr;
        const int hr0 = head_last ? k - 1 : 0, hm = head_last ? 1 : k;
        DFL_CK(head(c, c->h, hr0, hm, lg, AM_VERIFY));
        if (sampled) {
            SampleArgs sa{};
            sa.logits = c->logits;
            sa.M = hm;
            sa.row0 = hr0;
            sa.V = g.vocab;
            sa.ld = g.vocab;
            sa.st = c->st;
            sa.cnt = c->smp_cnt;
            DFL_LAUNCH_S(5, sa, launch_sample);
        }
    }
    return DFL_OK;
}

// ---- a long prefill pass: k (> 16) prompt rows at positions n..n+k-1 -------------------------------------
// Layer by layer over all k rows at once: the products on the tcgen05 tensor cores (tc_product), the
// row steps, q/k steps and attention over fp32 rows (attention in tiles of 16 rows), the gates as
// elementwise kernels. Sliding rings hold window + prefill_rows - 1 slots, so every row's window is
// still in its plane while the pass's later rows are appended (also for layers that read another
// layer's plane). The head runs on the last row only.
cudaError_t tc_product(dfl_ctx *c, const QMat &W, const float *x, int k, float *y) {
    c->launches += 3;   // weight expansion, row split, product
    return launch_tc_gemm(W.img, W.K, W.N, x, k, y, c->pf_scratch, &c->st->err, c->stream);
}

int prefill_long(dfl_ctx *c, int k, bool do_head, bool sampled) {
    const dfl_config &g = c->cfg;
    const int H = g.hidden, NL = g.n_layers, hd = g.head_dim, nq = g.n_heads, P = g.ple_dim;
    float *A = c->pf_a, *B = c->pf_b;   // two fp32 row buffers, alternately a step's input and output
    EmbedArgs ea{};
    ea.M = k;
    ea.H = H;
    ea.emb = c->emb.p;
    ea.scale = g.emb_scale;
    ea.st = c->st;
    ea.tokens = c->pf_tok;
    ea.x = c->pf_x;
    ea.ple = P ? c->ple_table.p : nullptr;
    ea.ple_w = NL * P;
    ea.ple_out = c->pf_ple;
    DFL_LAUNCH(launch_embed(ea, c->stream));
    RowArgs r0 = rows(c, k, c->pf_x);
    r0.w_next = c->tl[0].attn_norm.p;
    r0.out32 = A;
    DFL_LAUNCH(launch_rows(r0, c->stream));
    for (int l = 0; l < NL; ++l) {
        TLayer &L = c->tl[l];
        TLayer &O = c->tl[L.owner];
        const bool own = L.owner == l;
        const int nqkv = L.qkv.N;
        // attention block: A = normed rows
        DFL_CK(tc_product(c, L.qkv, A, k, B));
        QkArgs qa{};
        qa.M = k;
        qa.nq = nq;
        qa.nkv = L.nkv;
        qa.hd = hd;
        qa.qkv = B;
        qa.ldq = nqkv;
        qa.q_norm = L.q_norm.p;
        qa.k_norm = own ? L.k_norm.p : nullptr;
        qa.eps = g.eps;
        qa.rope = L.type == DFL_SLIDING ? c->rope_s : c->rope_f;
        qa.st = c->st;
        qa.q_out = A;
        qa.k_store = own ? L.K : nullptr;
        qa.v_store = own ? L.V : nullptr;
        qa.cap = L.cap;
        DFL_LAUNCH(launch_qk(qa, c->stream));
        AttnArgs aa{};
        aa.M = k;
        aa.nq = nq;
        aa.nkv = L.nkv;
        aa.hd = hd;
        aa.q = A;
        aa.kA = O.K;
        aa.vA = O.V;
        aa.capA = O.cap;
        aa.window = L.type == DFL_SLIDING ? g.window : 0;
        aa.mode = 0;
        aa.st = c->st;
        aa.scale = 1.0f / sqrtf((float)hd);
        aa.err = &c->st->err;
        // hundreds of 16-row tiles: the total work over all tiles, not one tile's latency, sets the time,
        // and clusters of 4 spend less of it in the merge than clusters of 16
        aa.max_cluster = std::min(c->attn_cluster, 4);
        aa.out32 = B;
        DFL_LAUNCH(launch_attn(aa, c->stream));
        DFL_CK(tc_product(c, L.o, B, k, A));
        RowArgs r1 = rows(c, k, c->pf_x);
        r1.y = A;
        r1.ldy = H;
        r1.w_post = L.post_attn_norm.p;
        r1.w_next = L.pre_ffn_norm.p;
        r1.out32 = B;
        DFL_LAUNCH(launch_rows(r1, c->stream));
        // FFN: B = normed rows
        DFL_CK(tc_product(c, L.gu, B, k, A));
        DFL_LAUNCH(launch_glu32(A, k, L.ffn, B, c->stream));
        DFL_CK(tc_product(c, L.d, B, k, A));
        const uint16_t *next = l + 1 < NL ? c->tl[l + 1].attn_norm.p : c->final_norm.p;
        int ti = 0;
        const bool tap = is_tap(g, l, &ti);
        RowArgs r2 = rows(c, k, c->pf_x);
        r2.y = A;
        r2.ldy = H;
        r2.w_post = L.post_ffn_norm.p;
        r2.out32 = B;
        if (P) {
            DFL_LAUNCH(launch_rows(r2, c->stream));   // out = x: the gate's input
            DFL_CK(tc_product(c, L.pg, B, k, A));
            DFL_LAUNCH(launch_silu_mul32(A, k, P, c->pf_ple + (size_t)l * P, NL * P, B, c->stream));
            DFL_CK(tc_product(c, L.pp, B, k, A));
            r2 = rows(c, k, c->pf_x);
            r2.y = A;
            r2.ldy = H;
            r2.w_post = L.ple_norm.p;
            r2.lambda = L.lambda;
            r2.out32 = B;
        }
        r2.w_next = next;
        if (tap) {
            r2.tap = c->taps;
            r2.ld_tap = c->TH;
            r2.tap_off = ti * H;
        }
        DFL_LAUNCH(launch_rows(r2, c->stream));
        std::swap(A, B);   // the next layer's input (B) is A again
    }
    if (do_head) {
        // the last row, final-normed, in the head's operand format
        DFL_LAUNCH(launch_act_pack(A + (size_t)(k - 1) * H, 1, H, c->h.f, c->h.s, c->stream));
        float *lg = (c->keep_logits || sampled) ? c->logits : nullptr;
        DFL_CK(head(c, c->h, 0, 1, lg, AM_VERIFY));
        if (sampled) {
            SampleArgs sa{};
            sa.logits = c->logits;
            sa.M = 1;
            sa.row0 = k - 1;
            sa.V = g.vocab;
            sa.ld = g.vocab;
            sa.st = c->st;
            sa.cnt = c->smp_cnt;
            DFL_LAUNCH(launch_sample(sa, c->stream));
        }
        c->have_logits = c->keep_logits || sampled;
    }
    return DFL_OK;
}

// A target pass of k rows at positions n..n+k-1 (the device counters are set beforehand).
int run_target(dfl_ctx *c, int k, bool do_head, bool sampled, bool head_last = false) {
    const bool early = c->stop_layer >= 0 && c->stop_layer < c->cfg.n_layers - 1;
    const uint64_t key = (1ull << 40) | (uint64_t)k | (uint64_t)do_head << 8 | (uint64_t)sampled << 9 |
                         (uint64_t)c->keep_logits << 10 | (uint64_t)head_last << 11 |
                         (uint64_t)(c->stop_layer + 1) << 12;
    const int rc = run_graph(c, key, [&] { return target_body(c, k, do_head, sampled, head_last); });
    if (rc) return rc;
    if (do_head && !early) c->have_logits = c->keep_logits || sampled;
    return DFL_OK;
}

// ---- draft context rows: fc of the taps, hidden norm, then each layer's key and value ---------------
// rows draft_n .. draft_n + r - 1 (device st->ctx_rows = r) into activation rows `row0..` of hctx.
// rows draft_n .. draft_n + st->ctx_rows - 1 become rows row0.. of hcat: RMSNorm_hidden(fc . taps)
int ctx_rows_prologue(dfl_ctx *c, int M, int row0) {
    const dfl_config &g = c->cfg;
    DFL_LAUNCH(launch_copy_taps(c->taps, c->TH, c->st, M, c->tapbuf.f, c->stream));
    DFL_CK(gemm(c, c->fc, c->tapbuf, 0, M, EPI_F32, c->y_fc, g.hidden));
    DFL_LAUNCH(launch_cast_rows(c->y_fc, g.hidden, M, g.hidden, c->d_hidden_norm.p, g.d_eps, c->hcat.f, c->hcat.s, row0,
                                c->st, 1, c->stream));
    return DFL_OK;
}

QkArgs draft_qk(dfl_ctx *c, int l) {
    const dfl_config &g = c->cfg;
    QkArgs qa{};
    qa.nq = g.d_heads;
    qa.nkv = g.d_kv_heads;
    qa.hd = g.d_head_dim;
    qa.qp = part_view(c, c->dl[l].qkv);
    qa.qkv_out = c->qkv;
    qa.ldq = c->dl[l].qkv.N;
    qa.q_norm = c->dl[l].q_norm.p;
    qa.k_norm = c->dl[l].k_norm.p;
    qa.eps = g.d_eps;
    qa.rope = c->rope_d;
    qa.st = c->st;
    return qa;
}

// a pass that only makes r <= 16 committed rows draft context
int run_ctx_only(dfl_ctx *c, int r) {
    const dfl_config &g = c->cfg;
    int rc = set_state(c, 0, nullptr, false, r, -1, nullptr);
    if (rc) return rc;
    rc = ctx_rows_prologue(c, kMaxRows, 0);
    if (rc) return rc;
    for (int l = 0; l < g.d_layers; ++l) {
        DLayer &D = c->dl[l];
        QkArgs qa = draft_qk(c, l);
        qa.M = kMaxRows;
        qa.row0 = 0;
        qa.pos_mode = 2;
        qa.live_from_ctx = 1;
        qa.k_store = D.K;
        qa.v_store = D.V;
        qa.cap = c->cap_draft;
        DFL_CK(gemm_qk(c, D.qkv, c->hcat, kMaxRows, qa));
    }
    c->draft_n += r;
    return DFL_OK;
}

int catch_up(dfl_ctx *c, int leave) {
    while (c->n - c->draft_n > leave) {
        const int r = std::min(kMaxRows, c->n - c->draft_n);
        const int rc = run_ctx_only(c, r);
        if (rc) return rc;
    }
    return DFL_OK;
}

int draft_body(dfl_ctx *c) {
    const dfl_config &g = c->cfg;
    const int H = g.hidden, B = g.block, F = c->ctx_fuse;
    if (F > 0) {
        const int rc = ctx_rows_prologue(c, F, B);
        if (rc) return rc;
    }
    EmbedArgs ea{};
    ea.M = B;
    ea.H = H;
    ea.emb = c->emb.p;
    ea.scale = g.d_emb_scale;
    ea.st = c->st;
    ea.use_draft = 1;
    ea.mask_token = g.mask_token;
    ea.x = c->x_d;
    DFL_LAUNCH_S(5, ea, launch_embed);
    RowArgs r0 = rows(c, B, c->x_d);
    r0.eps = g.d_eps;
    r0.w_next = c->dl[0].attn_norm.p;
    r0.outf = c->hcat.f;
    r0.outs = c->hcat.s;
    DFL_LAUNCH_S(5, r0, launch_rows);
    const int dq = g.d_heads, dhd = g.d_head_dim;
    for (int l = 0; l < g.d_layers; ++l) {
        DLayer &D = c->dl[l];
        QkArgs qb = draft_qk(c, l);
        qb.M = B;
        qb.pos_mode = 1;
        qb.q_out = c->q;
        qb.k_store = c->kB;
        qb.v_store = c->vB;
        qb.cap = 0;
        QkArgs qc = draft_qk(c, l);   // the fused context rows (after the block's rows)
        qc.M = F;
        qc.row0 = B;
        qc.pos_mode = 2;
        qc.live_from_ctx = 1;
        qc.k_store = D.K;
        qc.v_store = D.V;
        qc.cap = c->cap_draft;
        DFL_CK(gemm_qk(c, D.qkv, c->hcat, B + F, qb, F > 0 ? &qc : nullptr));
        AttnArgs aa{};
        aa.M = B;
        aa.nq = dq;
        aa.nkv = g.d_kv_heads;
        aa.hd = dhd;
        aa.q = c->q;
        aa.kA = D.K;
        aa.vA = D.V;
        aa.capA = c->cap_draft;
        aa.kB = c->kB;
        aa.vB = c->vB;
        aa.nB = B;
        aa.window = g.d_window;
        aa.mode = 1;
        aa.st = c->st;
        aa.scale = 1.0f / sqrtf((float)dhd);
        aa.err = &c->st->err;
        aa.max_cluster = c->attn_cluster;
        aa.outf = c->o.f;
        aa.outs = c->o.s;
        DFL_LAUNCH_S(3, aa, launch_attn);
        RowArgs r1 = rows(c, B, c->x_d);
        r1.eps = g.d_eps;
        r1.y_out = c->y;
        r1.w_next = D.ffn_norm.p;
        r1.outf = c->hb.f;
        r1.outs = c->hb.s;
        DFL_CK(gemm_rows(c, D.o, c->o, B, r1));
        DFL_CK(gemm(c, D.gu, c->hb, 0, B, EPI_GLU, nullptr, 0, &c->a));
        RowArgs r2 = rows(c, B, c->x_d);
        r2.eps = g.d_eps;
        r2.y_out = c->y;
        r2.w_next = l + 1 < g.d_layers ? c->dl[l + 1].attn_norm.p : c->d_final_norm.p;
        const Act &nxt = l + 1 < g.d_layers ? c->hcat : c->hb;
        r2.outf = nxt.f;
        r2.outs = nxt.s;
        DFL_CK(gemm_rows(c, D.d, c->a, B, r2));
    }
    float *lg = c->keep_logits ? c->dlogits : nullptr;
    DFL_CK(head(c, c->hb, 1, B - 1, lg, AM_DRAFT));
    return DFL_OK;
}

// Draft block at positions n..n+block-1; first makes the r <= ctx_fuse committed rows not yet in the
// draft context into context (fused into the same pass).
int run_draft(dfl_ctx *c, int last_tok) {
    const int r = c->n - c->draft_n;
    int rc = set_state(c, c->cfg.block, nullptr, false, r, last_tok, nullptr);
    if (rc) return rc;
    rc = run_graph(c, (2ull << 40) | (uint64_t)c->keep_logits, [&] { return draft_body(c); });
    if (rc) return rc;
    c->have_dlogits = c->keep_logits;
    c->draft_n += r;
    return DFL_OK;
}



// Read the device counters (synchronises the stream). A bounded wait that gave up in any pass since
// the last read is reported as DFL_E_TIMEOUT: the error bits are cleared, the draft context falls back
// to the rows confirmed by the last good read (the rows made context since then are made again by the
// next draft block), and the caller restores its own counters. Committed planes, taps and positions
// are untouched by a failed pass (it writes only rows past the committed positions).
int read_state(dfl_ctx *c, DevState *out) {
    DFL_CK(cudaMemcpyAsync(out, c->st, sizeof(DevState), cudaMemcpyDeviceToHost, c->stream));
    DFL_CK(cudaStreamSynchronize(c->stream));
    if (out->err & kErrWaitTimeout) {
        DFL_CK(cudaMemsetAsync(&c->st->err, 0, sizeof(int), c->stream));
        // a pass that gave up may leave arrival counters short of their reset: start them from zero
        DFL_CK(cudaMemsetAsync(c->counters_begin, 0, c->counters_bytes, c->stream));
        DFL_CK(cudaStreamSynchronize(c->stream));
        c->draft_n = std::min(c->draft_n_ok, c->n);
        c->draft_n_ok = c->draft_n;
        c->draft_at = -1;
        return fail(c, DFL_E_TIMEOUT, "a kernel gave up waiting for its asynchronous copies (bounded wait)");
    }
    c->draft_n_ok = c->draft_n;
    return DFL_OK;
}

int check_tokens(dfl_ctx *c, const int32_t *t, int n) {
    for (int i = 0; i < n; ++i)
        if (t[i] < 0 || t[i] >= c->cfg.vocab) return fail(c, DFL_E_INVALID_ARG, "token id out of range");
    return DFL_OK;
}

int ready(dfl_ctx *c) {
    if (c->needs_restore)
        return fail(c, DFL_E_STATE, "a failed prefill may have overwritten ring slots of the held positions: restore a snapshot");
    auto chk = [&](bool ok, const char *what) { return ok ? DFL_OK : fail(c, DFL_E_STATE, std::string("tensor not loaded: ") + what); };
    int rc;
    if ((rc = chk(c->emb.loaded && c->head.loaded && c->final_norm.loaded, "emb/head/final_norm"))) return rc;
    if (c->cfg.ple_dim && (rc = chk(c->ple_table.loaded, "ple_table"))) return rc;
    for (size_t l = 0; l < c->tl.size(); ++l) {
        const TLayer &L = c->tl[l];
        bool ok = L.qkv.loaded && L.o.loaded && L.gu.loaded && L.d.loaded && L.attn_norm.loaded && L.q_norm.loaded &&
                  L.post_attn_norm.loaded && L.pre_ffn_norm.loaded && L.post_ffn_norm.loaded;
        if (L.owner == (int)l) ok = ok && L.k_norm.loaded;
        if (c->cfg.ple_dim) ok = ok && L.pg.loaded && L.pp.loaded && L.ple_norm.loaded && L.lam.loaded;
        if ((rc = chk(ok, ("t" + std::to_string(l) + ".*").c_str()))) return rc;
    }
    if ((rc = chk(c->fc.loaded && c->d_hidden_norm.loaded && c->d_final_norm.loaded, "d.fc/d.hidden_norm/d.final_norm")))
        return rc;
    for (size_t l = 0; l < c->dl.size(); ++l) {
        const DLayer &D = c->dl[l];
        const bool ok = D.qkv.loaded && D.o.loaded && D.gu.loaded && D.d.loaded && D.attn_norm.loaded &&
                        D.q_norm.loaded && D.k_norm.loaded && D.ffn_norm.loaded;
        if ((rc = chk(ok, ("d" + std::to_string(l) + ".*").c_str()))) return rc;
    }
    return DFL_OK;
}

size_t snapshot_size(const dfl_ctx *c, int n, int draft_n) {
    const dfl_config &g = c->cfg;
    size_t b = sizeof(SnapHeader);
    for (int l = 0; l < g.n_layers; ++l) {
        const TLayer &L = c->tl[l];
        if (L.owner != l) continue;
        const size_t row = (size_t)L.nkv * g.head_dim * 4;
        const size_t rows = L.type == DFL_SLIDING ? (size_t)L.cap : (size_t)n;
        b += 2 * rows * row;
    }
    b += (size_t)g.d_layers * 2 * c->cap_draft * g.d_kv_heads * g.d_head_dim * 4;
    b += (size_t)(n - draft_n) * c->TH * 4;
    return b;
}

}  // namespace

// =====================================================================================================
// C ABI
// =====================================================================================================
extern "C" {

int dfl_required_bytes(const dfl_config *cfg, dfl_sizes *out) {
    if (!cfg || !out) return DFL_E_INVALID_ARG;
    if (!validate(cfg).empty()) return DFL_E_INVALID_ARG;
    dfl_ctx tmp;
    tmp.cfg = *cfg;
    Arena W, S, X;
    plan(&tmp, W, S, X);
    out->weights_bytes = W.off;
    out->state_bytes = S.off;
    out->workspace_bytes = X.off;
    return DFL_OK;
}

int dfl_init(const dfl_config *cfg, const dfl_buffers *buf, void *stream, dfl_ctx **out) {
    if (!cfg || !buf || !out) return DFL_E_INVALID_ARG;
    *out = nullptr;
    if (!validate(cfg).empty()) return DFL_E_INVALID_ARG;
    if (!buf->weights || !buf->state || !buf->workspace) return DFL_E_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(buf->weights) | reinterpret_cast<uintptr_t>(buf->state) |
         reinterpret_cast<uintptr_t>(buf->workspace)) & 255)
        return DFL_E_INVALID_ARG;
    dfl_ctx *c = new dfl_ctx();
    c->cfg = *cfg;
    c->stream = static_cast<cudaStream_t>(stream);
    Arena W, S, X;
    W.base = static_cast<uint8_t *>(buf->weights);
    S.base = static_cast<uint8_t *>(buf->state);
    X.base = static_cast<uint8_t *>(buf->workspace);
    plan(c, W, S, X);
    auto bail = [&](cudaError_t e, const char *what) {
        delete c;
        (void)e;
        (void)what;
        return DFL_E_CUDA;
    };
    cudaError_t e;
    if ((e = cudaMemsetAsync(buf->state, 0, S.off, c->stream)) != cudaSuccess) return bail(e, "memset state");
    if ((e = cudaMemsetAsync(c->counters_begin, 0, c->counters_bytes, c->stream)) != cudaSuccess) return bail(e, "memset");
    const dfl_config &g = c->cfg;
    if ((e = launch_rope_table(c->rope_s, c->rope_rows, g.head_dim, g.rope_base_sliding, c->stream)) != cudaSuccess ||
        (e = launch_rope_table(c->rope_f, c->rope_rows, g.head_dim, g.rope_base_full, c->stream)) != cudaSuccess ||
        (e = launch_rope_table(c->rope_d, c->rope_rows, g.d_head_dim, g.d_rope_base, c->stream)) != cudaSuccess)
        return bail(e, "rope table");
    if ((e = attn_prepare(g.head_dim)) != cudaSuccess || (e = attn_prepare(g.d_head_dim)) != cudaSuccess)
        return bail(e, "attention setup");
    if ((e = cudaStreamSynchronize(c->stream)) != cudaSuccess) return bail(e, "sync");
    c->launches = 3;   // the rope tables
    *out = c;
    return DFL_OK;
}

int dfl_load_tensor(dfl_ctx *c, const char *name, const void *src, size_t bytes) {
    if (!c) return DFL_E_INVALID_ARG;
    if (!name || !src) return fail(c, DFL_E_INVALID_ARG, "null name or source");
    const dfl_config &g = c->cfg;
    const std::string s(name);
    QMat *m = nullptr;
    Vec *v = nullptr;
    TLayer *tlay = nullptr;
    auto field = [&](const std::string &f, int layer, bool draft) -> bool {
        if (draft) {
            DLayer &D = c->dl[layer];
            if (f == "attn_norm") v = &D.attn_norm;
            else if (f == "q_norm") v = &D.q_norm;
            else if (f == "k_norm") v = &D.k_norm;
            else if (f == "ffn_norm") v = &D.ffn_norm;
            else if (f == "wqkv") m = &D.qkv;
            else if (f == "wo") m = &D.o;
            else if (f == "wgu") m = &D.gu;
            else if (f == "wd") m = &D.d;
            else return false;
            return true;
        }
        TLayer &L = c->tl[layer];
        const bool own = L.owner == layer;
        tlay = &L;
        if (f == "attn_norm") v = &L.attn_norm;
        else if (f == "q_norm") v = &L.q_norm;
        else if (f == "k_norm" && own) v = &L.k_norm;
        else if (f == "post_attn_norm") v = &L.post_attn_norm;
        else if (f == "pre_ffn_norm") v = &L.pre_ffn_norm;
        else if (f == "post_ffn_norm") v = &L.post_ffn_norm;
        else if (f == "ple_norm" && g.ple_dim) v = &L.ple_norm;
        else if (f == "lambda" && g.ple_dim) v = &L.lam;
        else if ((f == "wqkv" && own) || (f == "wq" && !own)) m = &L.qkv;
        else if (f == "wo") m = &L.o;
        else if (f == "wgu") m = &L.gu;
        else if (f == "wd") m = &L.d;
        else if (f == "wple_g" && g.ple_dim) m = &L.pg;
        else if (f == "wple_p" && g.ple_dim) m = &L.pp;
        else return false;
        return true;
    };
    bool ok = false;
    if (s == "emb") v = &c->emb, ok = true;
    else if (s == "head") m = &c->head, ok = true;
    else if (s == "final_norm") v = &c->final_norm, ok = true;
    else if (s == "ple_table" && g.ple_dim) v = &c->ple_table, ok = true;
    else if (s == "d.fc") m = &c->fc, ok = true;
    else if (s == "d.hidden_norm") v = &c->d_hidden_norm, ok = true;
    else if (s == "d.final_norm") v = &c->d_final_norm, ok = true;
    else if (s.size() > 2 && (s[0] == 't' || s[0] == 'd') && isdigit((unsigned char)s[1])) {
        const size_t dot = s.find('.');
        if (dot != std::string::npos) {
            const int layer = atoi(s.substr(1, dot - 1).c_str());
            const bool draft = s[0] == 'd';
            if (layer >= 0 && layer < (draft ? g.d_layers : g.n_layers)) ok = field(s.substr(dot + 1), layer, draft);
        }
    }
    if (!ok) return fail(c, DFL_E_INVALID_ARG, "unknown tensor name: " + s);
    if (m) {
        const size_t want = m->q41 ? (size_t)m->N * (m->K / 32) * 20 : (size_t)m->N * m->K * 2;
        if (bytes != want) return fail(c, DFL_E_INVALID_ARG, s + ": expected " + std::to_string(want) + " bytes");
        if (m->q41) DFL_LAUNCH(launch_pack_q41(static_cast<const uint8_t *>(src), m->K, m->N, m->img, c->stream));
        else DFL_LAUNCH(launch_pack_bf16(static_cast<const uint16_t *>(src), m->K, m->N, m->img, c->stream));
        m->loaded = true;
        return DFL_OK;
    }
    if (bytes != v->n * 2) return fail(c, DFL_E_INVALID_ARG, s + ": expected " + std::to_string(v->n * 2) + " bytes");
    DFL_CK(cudaMemcpyAsync(v->p, src, bytes, cudaMemcpyDeviceToDevice, c->stream));
    if (tlay && v == &tlay->lam) {
        uint16_t b = 0;
        DFL_CK(cudaMemcpyAsync(&b, src, 2, cudaMemcpyDeviceToHost, c->stream));
        DFL_CK(cudaStreamSynchronize(c->stream));
        uint32_t u = uint32_t(b) << 16;
        float f;
        memcpy(&f, &u, 4);
        tlay->lambda = f;
    }
    v->loaded = true;
    return DFL_OK;
}

int dfl_prefill(dfl_ctx *c, const int32_t *tokens, int n, const dfl_sampling *s, int32_t *next_tok) {
    NvtxRange nvtx("dfl_prefill");
    if (!c) return DFL_E_INVALID_ARG;
    if (!tokens || n < 1) return fail(c, DFL_E_INVALID_ARG, "prefill needs at least one token");
    if (c->pending) return fail(c, DFL_E_STATE, "a verify is pending: commit it first");
    if (c->draft_only) return fail(c, DFL_E_STATE, "context holds draft-only rows");
    if ((long)c->n + n > c->cfg.max_ctx) return fail(c, DFL_E_CAPACITY, "prefill exceeds max_ctx");
    int rc = ready(c);
    if (rc) return rc;
    if ((rc = check_tokens(c, tokens, n))) return rc;
    const bool sampled = s && s->temperature > 0.f;
    const int n_start = c->n;
    // On an error after the first pass was enqueued none of the rows counts. The passes already run
    // may have written ring slots that positions held still need (more rows than a ring's slack, or
    // rows of the draft context's window), so the context also refuses passes until a restore.
    auto failed = [&](int rc_) {
        c->n = n_start;
        c->draft_n = std::min(c->draft_n, n_start);
        c->draft_n_ok = std::min(c->draft_n_ok, c->draft_n);
        c->draft_at = -1;
        c->needs_restore = n_start > 0;   // an empty context has no slot to lose
        return rc_;
    };
    int done = 0;
    const int PF = c->cfg.prefill_rows;
    while (done < n) {
        // long passes while at least 128 rows remain (prefill_rows > 0), then passes of up to 16 rows
        const bool longp = PF > 0 && n - done >= 128;
        const int k = longp ? std::min(PF, n - done) : std::min(kMaxRows, n - done);
        const bool last = done + k == n;
        if ((rc = set_state(c, k, tokens + done, false, 0, -1, s))) return failed(rc);
        if (longp) {
            if (cudaMemcpyAsync(c->pf_tok, tokens + done, sizeof(int32_t) * k, cudaMemcpyHostToDevice, c->stream) !=
                cudaSuccess)
                return failed(fail(c, DFL_E_CUDA, "prefill token copy failed"));
            if ((rc = prefill_long(c, k, last, sampled))) return failed(rc);
        } else if ((rc = run_target(c, k, last, sampled, true))) {
            return failed(rc);
        }
        c->n += k;
        done += k;
    }
    if ((rc = catch_up(c, 0))) return failed(rc);
    DevState hs;
    if ((rc = read_state(c, &hs))) return failed(rc);
    if (next_tok) *next_tok = hs.target[0];   // the head ran on the last row only
    c->last_k = 1;                            // logits of that row
    c->draft_at = -1;
    return DFL_OK;
}

int dfl_draft_block(dfl_ctx *c, int32_t last_tok, int32_t *proposals) {
    NvtxRange nvtx("dfl_draft_block");
    if (!c) return DFL_E_INVALID_ARG;
    if (c->pending) return fail(c, DFL_E_STATE, "a verify is pending: commit it first");
    if (last_tok < 0 || last_tok >= c->cfg.vocab) return fail(c, DFL_E_INVALID_ARG, "token id out of range");
    if ((long)c->n + c->cfg.block > c->cfg.max_ctx + kMaxRows) return fail(c, DFL_E_CAPACITY, "block past max_ctx");
    int rc = ready(c);
    if (rc) return rc;
    if ((rc = catch_up(c, c->ctx_fuse))) return rc;
    if ((rc = run_draft(c, last_tok))) return rc;
    c->draft_at = c->n;
    if (proposals) {
        DevState hs;
        if ((rc = read_state(c, &hs))) return rc;
        for (int i = 0; i < c->cfg.block - 1; ++i) proposals[i] = hs.props[i];
    }
    return DFL_OK;
}

int dfl_verify_block(dfl_ctx *c, const int32_t *rows_in, int k, const dfl_sampling *s, int32_t *target_tok,
                     int32_t *accepted) {
    NvtxRange nvtx("dfl_verify_block");
    if (!c) return DFL_E_INVALID_ARG;
    if (c->pending) return fail(c, DFL_E_STATE, "a verify is pending: commit it first");
    if (c->draft_only) return fail(c, DFL_E_STATE, "context holds draft-only rows");
    if (k < 1 || k > kMaxRows) return fail(c, DFL_E_UNSUPPORTED, "k must be 1..16");
    if ((long)c->n + k > c->cfg.max_ctx) return fail(c, DFL_E_CAPACITY, "verify exceeds max_ctx");
    int rc = ready(c);
    if (rc) return rc;
    if (rows_in) {
        if ((rc = check_tokens(c, rows_in, k))) return rc;
    } else {
        if (c->draft_at != c->n) return fail(c, DFL_E_STATE, "rows = NULL needs a draft block at this position");
        if (k > c->cfg.block) return fail(c, DFL_E_INVALID_ARG, "k exceeds the draft block");
    }
    const bool sampled = s && s->temperature > 0.f;
    if ((rc = set_state(c, k, rows_in, rows_in == nullptr, 0, -1, s))) return rc;
    if ((rc = run_target(c, k, true, sampled))) return rc;
    DevState hs;
    if ((rc = read_state(c, &hs))) return rc;
    if (target_tok)
        for (int i = 0; i < k; ++i) target_tok[i] = hs.target[i];
    if (accepted) *accepted = hs.accepted;
    c->pending = k;
    c->last_k = k;
    c->last_accepted = hs.accepted;
    for (int i = 0; i < k; ++i) c->last_target[i] = hs.target[i];
    return DFL_OK;
}

int dfl_commit_verify_rows(dfl_ctx *c, int keep) {
    if (!c) return DFL_E_INVALID_ARG;
    if (!c->pending) return fail(c, DFL_E_STATE, "no pending verify");
    if (keep == DFL_KEEP_ACCEPTED) keep = std::min(c->last_accepted + 1, c->pending);
    if (keep < 0 || keep > c->pending) return fail(c, DFL_E_INVALID_ARG, "keep must be 0..k");
    c->n += keep;
    c->pending = 0;
    c->draft_at = -1;
    return DFL_OK;
}

int dfl_commit_accepted(dfl_ctx *c, int max_keep, int32_t stop_token, int32_t *kept, int32_t *stopped) {
    if (!c) return DFL_E_INVALID_ARG;
    if (!c->pending) return fail(c, DFL_E_STATE, "no pending verify");
    if (max_keep < 0) return fail(c, DFL_E_INVALID_ARG, "max_keep must be >= 0");
    int keep = std::min(std::min(c->last_accepted + 1, c->pending), max_keep);
    int stop = 0;
    if (stop_token >= 0)
        for (int i = 0; i < keep; ++i)
            if (c->last_target[i] == stop_token) {   // token i is emitted; the row it would feed is not kept
                keep = i + 1;
                stop = 1;
                break;
            }
    const int rc = dfl_commit_verify_rows(c, keep);
    if (rc == DFL_OK) {
        if (kept) *kept = keep;
        if (stopped) *stopped = stop;
    }
    return rc;
}

int64_t dfl_snapshot_bytes(const dfl_ctx *c) {
    if (!c) return -1;
    return (int64_t)snapshot_size(c, c->n, c->draft_n);
}

int dfl_snapshot(dfl_ctx *c, void *dst, size_t bytes) {
    NvtxRange nvtx("dfl_snapshot");
    if (!c) return DFL_E_INVALID_ARG;
    if (c->pending) return fail(c, DFL_E_STATE, "snapshot needs the committed state");
    if (c->needs_restore) return fail(c, DFL_E_STATE, "a failed prefill left the state unusable: restore first");
    if (!dst) return fail(c, DFL_E_INVALID_ARG, "null destination");
    const size_t need = snapshot_size(c, c->n, c->draft_n);
    if (bytes < need) return fail(c, DFL_E_INVALID_ARG, "snapshot buffer too small");
    const dfl_config &g = c->cfg;
    SnapHeader hdr{};
    hdr.magic = kSnapMagic;
    hdr.version = 1;
    hdr.cfg_hash = fnv1a(&c->cfg, sizeof(dfl_config));
    hdr.n = c->n;
    hdr.draft_n = c->draft_n;
    hdr.bytes = need;
    uint8_t *d = static_cast<uint8_t *>(dst);
    DFL_CK(cudaMemcpyAsync(d, &hdr, sizeof hdr, cudaMemcpyHostToDevice, c->stream));
    size_t off = sizeof hdr;
    for (int l = 0; l < g.n_layers; ++l) {
        const TLayer &L = c->tl[l];
        if (L.owner != l) continue;
        const size_t row = (size_t)L.nkv * g.head_dim * 4;
        const size_t rows = L.type == DFL_SLIDING ? (size_t)L.cap : (size_t)c->n;
        DFL_CK(cudaMemcpyAsync(d + off, L.K, rows * row, cudaMemcpyDeviceToDevice, c->stream));
        off += rows * row;
        DFL_CK(cudaMemcpyAsync(d + off, L.V, rows * row, cudaMemcpyDeviceToDevice, c->stream));
        off += rows * row;
    }
    const size_t dbytes = (size_t)c->cap_draft * g.d_kv_heads * g.d_head_dim * 4;
    for (int l = 0; l < g.d_layers; ++l) {
        DFL_CK(cudaMemcpyAsync(d + off, c->dl[l].K, dbytes, cudaMemcpyDeviceToDevice, c->stream));
        off += dbytes;
        DFL_CK(cudaMemcpyAsync(d + off, c->dl[l].V, dbytes, cudaMemcpyDeviceToDevice, c->stream));
        off += dbytes;
    }
    const size_t tb = (size_t)(c->n - c->draft_n) * c->TH * 4;
    if (tb) DFL_CK(cudaMemcpyAsync(d + off, c->taps + (size_t)c->draft_n * c->TH, tb, cudaMemcpyDeviceToDevice, c->stream));
    DFL_CK(cudaStreamSynchronize(c->stream));   // the header came from host memory on this stack
    return DFL_OK;
}

int dfl_restore(dfl_ctx *c, const void *src, size_t bytes) {
    NvtxRange nvtx("dfl_restore");
    if (!c) return DFL_E_INVALID_ARG;
    if (c->pending) return fail(c, DFL_E_STATE, "restore needs the committed state");
    if (!src || bytes < sizeof(SnapHeader)) return fail(c, DFL_E_INVALID_ARG, "snapshot too small");
    SnapHeader hdr;
    DFL_CK(cudaMemcpyAsync(&hdr, src, sizeof hdr, cudaMemcpyDeviceToHost, c->stream));
    DFL_CK(cudaStreamSynchronize(c->stream));
    const dfl_config &g = c->cfg;
    if (hdr.magic != kSnapMagic || hdr.version != 1) return fail(c, DFL_E_INVALID_ARG, "not a snapshot");
    if (hdr.cfg_hash != fnv1a(&c->cfg, sizeof(dfl_config))) return fail(c, DFL_E_INVALID_ARG, "snapshot of another configuration");
    if (hdr.n < 0 || hdr.n > g.max_ctx || hdr.draft_n < 0 || hdr.draft_n > hdr.n)
        return fail(c, DFL_E_INVALID_ARG, "corrupt snapshot header");
    const size_t need = snapshot_size(c, hdr.n, hdr.draft_n);
    if (hdr.bytes != need || bytes < need) return fail(c, DFL_E_INVALID_ARG, "snapshot size mismatch");
    const uint8_t *s = static_cast<const uint8_t *>(src);
    size_t off = sizeof hdr;
    for (int l = 0; l < g.n_layers; ++l) {
        const TLayer &L = c->tl[l];
        if (L.owner != l) continue;
        const size_t row = (size_t)L.nkv * g.head_dim * 4;
        const size_t rows = L.type == DFL_SLIDING ? (size_t)L.cap : (size_t)hdr.n;
        DFL_CK(cudaMemcpyAsync(L.K, s + off, rows * row, cudaMemcpyDeviceToDevice, c->stream));
        off += rows * row;
        DFL_CK(cudaMemcpyAsync(L.V, s + off, rows * row, cudaMemcpyDeviceToDevice, c->stream));
        off += rows * row;
    }
    const size_t dbytes = (size_t)c->cap_draft * g.d_kv_heads * g.d_head_dim * 4;
    for (int l = 0; l < g.d_layers; ++l) {
        DFL_CK(cudaMemcpyAsync(c->dl[l].K, s + off, dbytes, cudaMemcpyDeviceToDevice, c->stream));
        off += dbytes;
        DFL_CK(cudaMemcpyAsync(c->dl[l].V, s + off, dbytes, cudaMemcpyDeviceToDevice, c->stream));
        off += dbytes;
    }
    const size_t tb = (size_t)(hdr.n - hdr.draft_n) * c->TH * 4;
    if (tb) DFL_CK(cudaMemcpyAsync(c->taps + (size_t)hdr.draft_n * c->TH, s + off, tb, cudaMemcpyDeviceToDevice, c->stream));
    c->n = hdr.n;
    c->draft_n = hdr.draft_n;
    c->draft_n_ok = hdr.draft_n;
    c->draft_at = -1;
    c->draft_only = false;
    c->needs_restore = false;
    return DFL_OK;
}

int dfl_kv_widths(const dfl_ctx *c, int32_t *out) {
    if (!c || !out) return DFL_E_INVALID_ARG;
    for (int l = 0; l < c->cfg.n_layers; ++l)
        out[l] = c->tl[l].owner == l ? 2 * c->tl[l].nkv * c->cfg.head_dim : 0;
    return DFL_OK;
}

int64_t dfl_positions_held(const dfl_ctx *c) { return c ? c->n : -1; }

int dfl_set_option(dfl_ctx *c, int option, int value) {
    if (!c) return DFL_E_INVALID_ARG;
    if (option == DFL_OPT_KEEP_LOGITS) c->keep_logits = value != 0;
    else if (option == DFL_OPT_GRAPHS) c->use_graphs = value != 0;
    else if (option == DFL_OPT_STOP_LAYER) c->stop_layer = value;
    else if (option == DFL_OPT_PROFILE) {
        DFL_CK(cudaStreamSynchronize(c->stream));
        c->profile = value != 0;
        c->recs.clear();
        for (int i = 0; i < kProfClasses; ++i) c->prof_ms[i] = c->prof_bytes[i] = 0, c->prof_n[i] = 0;
    }
    else if (option == DFL_OPT_TEST_STALL) c->test_stall = value != 0;
    else if (option == DFL_OPT_PLE_SPLIT) {
        if ((value != 0) != c->ple_split) {
            DFL_CK(cudaStreamSynchronize(c->stream));
            for (auto &kv : c->graphs) cudaGraphExecDestroy(kv.second.exec);   // captured the other way
            c->graphs.clear();
            c->ple_split = value != 0;
        }
    }
    else if (option == DFL_OPT_FUSE_STEPS) {
        if ((value != 0) != c->fuse_steps) {
            DFL_CK(cudaStreamSynchronize(c->stream));
            for (auto &kv : c->graphs) cudaGraphExecDestroy(kv.second.exec);   // captured the other way
            c->graphs.clear();
            c->fuse_steps = value != 0;
        }
    }
    else if (option == DFL_OPT_ATTN_CLUSTER) {
        if (value != 4 && value != 8 && value != 16)
            return fail(c, DFL_E_INVALID_ARG, "attention cluster must be 4, 8 or 16");
        if (value != c->attn_cluster) {
            DFL_CK(cudaStreamSynchronize(c->stream));
            for (auto &kv : c->graphs) cudaGraphExecDestroy(kv.second.exec);   // captured with the old size
            c->graphs.clear();
            c->attn_cluster = value;
        }
    }
    else return fail(c, DFL_E_INVALID_ARG, "unknown option");
    return DFL_OK;
}

int dfl_read_logits(dfl_ctx *c, int which, float *dst, int rows) {
    if (!c || !dst) return DFL_E_INVALID_ARG;
    const int V = c->cfg.vocab;
    if (which == 0) {
        if (!c->have_logits) return fail(c, DFL_E_STATE, "no verify logits kept");
        if (rows < 1 || rows > c->last_k) return fail(c, DFL_E_INVALID_ARG, "rows out of range");
        DFL_CK(cudaMemcpyAsync(dst, c->logits, (size_t)rows * V * 4, cudaMemcpyDeviceToHost, c->stream));
    } else if (which == 1) {
        if (!c->have_dlogits) return fail(c, DFL_E_STATE, "no draft logits kept");
        if (rows < 1 || rows > c->cfg.block - 1) return fail(c, DFL_E_INVALID_ARG, "rows out of range");
        DFL_CK(cudaMemcpyAsync(dst, c->dlogits, (size_t)rows * V * 4, cudaMemcpyDeviceToHost, c->stream));
    } else {
        return fail(c, DFL_E_INVALID_ARG, "which must be 0 or 1");
    }
    DFL_CK(cudaStreamSynchronize(c->stream));
    return DFL_OK;
}

int dfl_read_taps(dfl_ctx *c, int pos0, int rows, float *dst) {
    if (!c || !dst) return DFL_E_INVALID_ARG;
    if (pos0 < 0 || rows < 1 || pos0 + rows > c->cfg.max_ctx + kMaxRows) return fail(c, DFL_E_INVALID_ARG, "rows out of range");
    DFL_CK(cudaMemcpyAsync(dst, c->taps + (size_t)pos0 * c->TH, (size_t)rows * c->TH * 4, cudaMemcpyDeviceToHost, c->stream));
    DFL_CK(cudaStreamSynchronize(c->stream));
    return DFL_OK;
}

int dfl_draft_append_taps(dfl_ctx *c, const void *src, int rows) {
    NvtxRange nvtx("dfl_draft_append_taps");
    if (!c) return DFL_E_INVALID_ARG;
    if (!src || rows < 1) return fail(c, DFL_E_INVALID_ARG, "bad taps");
    if (c->pending) return fail(c, DFL_E_STATE, "a verify is pending");
    if ((long)c->n + rows > c->cfg.max_ctx) return fail(c, DFL_E_CAPACITY, "taps exceed max_ctx");
    int rc = ready(c);
    if (rc) return rc;
    DFL_CK(cudaMemcpyAsync(c->taps + (size_t)c->n * c->TH, src, (size_t)rows * c->TH * 4, cudaMemcpyDeviceToDevice,
                           c->stream));
    c->n += rows;
    c->draft_only = true;
    c->draft_at = -1;
    return catch_up(c, 0);
}

int dfl_debug_read(dfl_ctx *c, const char *name, void *dst, size_t bytes) {
    if (!c || !name || !dst) return DFL_E_INVALID_ARG;
    const std::string s(name);
    const void *src = nullptr;
    size_t have = 0;
    const size_t R = kMaxRows, H = c->cfg.hidden;
    if (s == "x") src = c->x, have = R * H * 4;
    else if (s == "y") src = c->y, have = R * H * 4;
    else if (s == "qkv") src = c->qkv, have = R * c->qkv_max * 4;
    else if (s == "q") src = c->q, have = R * std::max(c->cfg.n_heads * c->cfg.head_dim, c->cfg.d_heads * c->cfg.d_head_dim) * 4;
    else if (s == "x_d") src = c->x_d, have = R * H * 4;
    else if (s.size() > 1 && (s[0] == 'k' || s[0] == 'v') && isdigit((unsigned char)s[1])) {
        size_t used = 0;
        const int l = std::stoi(s.substr(1), &used);
        if (used != s.size() - 1 || l < 0 || l >= c->cfg.n_layers) return fail(c, DFL_E_INVALID_ARG, "bad layer in " + s);
        const TLayer &L = c->tl[l];
        if (L.owner != l) return fail(c, DFL_E_INVALID_ARG, s + ": a KV-shared layer holds no plane");
        src = s[0] == 'k' ? L.K : L.V;
        have = (size_t)L.cap * L.nkv * c->cfg.head_dim * 4;
    }
    else return fail(c, DFL_E_INVALID_ARG, "unknown buffer " + s);
    if (bytes > have) return fail(c, DFL_E_INVALID_ARG, "read past the buffer");
    DFL_CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, c->stream));
    DFL_CK(cudaStreamSynchronize(c->stream));
    return DFL_OK;
}

int dfl_plant_proposals(dfl_ctx *c, const int32_t *dev_table, int table_len) {
    if (!c) return DFL_E_INVALID_ARG;
    if (!dev_table) return fail(c, DFL_E_INVALID_ARG, "null table");
    if (c->draft_at != c->n || c->pending) return fail(c, DFL_E_STATE, "planting needs a draft block at this position");
    if ((long)c->n + c->cfg.block > table_len) return fail(c, DFL_E_INVALID_ARG, "table shorter than the block's positions");
    DFL_LAUNCH(launch_plant(c->st, dev_table, c->cfg.block - 1, c->stream));
    return DFL_OK;
}

int64_t dfl_launch_count(const dfl_ctx *c) { return c ? c->launches : -1; }

int dfl_profile_read(dfl_ctx *c, int cls, int64_t *launches, double *ms, double *bytes) {
    if (!c || cls < 0 || cls >= kProfClasses) return DFL_E_INVALID_ARG;
    DFL_CK(cudaStreamSynchronize(c->stream));
    if (launches) *launches = c->prof_n[cls];
    if (ms) *ms = c->prof_ms[cls];
    if (bytes) *bytes = c->prof_bytes[cls];
    return DFL_OK;
}

const char *dfl_last_error(const dfl_ctx *c) { return c ? c->err.c_str() : "null context"; }

void dfl_destroy(dfl_ctx *c) {
    if (!c) return;
    if (c->stream) cudaStreamSynchronize(c->stream);
    for (auto &kv : c->graphs) cudaGraphExecDestroy(kv.second.exec);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    delete c;
}

int64_t dfl_q41_image_bytes(int K, int N) {
    if (K < 32 || K % 32 || N < 32 || N % 32) return -1;
    return (int64_t)q41_image_bytes(K, N);
}

int dfl_q41_pack(const void *src, int K, int N, void *img, void *stream) {
    if (!src || !img || K < 32 || K % 32 || N < 32 || N % 32) return DFL_E_INVALID_ARG;
    return launch_pack_q41(static_cast<const uint8_t *>(src), K, N, static_cast<uint8_t *>(img),
                           static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFL_OK : DFL_E_CUDA;
}

int64_t dfl_act_bytes(int M, int K) {
    if (M < 1 || M > kMaxRows || K < 16 || K % 16) return -1;
    return (int64_t)(act_words(K) * 4 + act_sums(K) * 4);
}

int dfl_act_pack(const float *x, int M, int K, void *act, void *stream) {
    if (!x || !act || dfl_act_bytes(M, K) < 0) return DFL_E_INVALID_ARG;
    uint32_t *f = static_cast<uint32_t *>(act);
    float *sums = reinterpret_cast<float *>(f + act_words(K));
    return launch_act_pack(x, M, K, f, sums, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFL_OK : DFL_E_CUDA;
}

// scratch = a 256-byte header (the error word at offset 0), the arrival counters (N/32 ints, rounded up
// to 256 bytes), then the segment partials
constexpr size_t kScratchHeader = 256;
int64_t dfl_q41_gemm_scratch_bytes(int K, int N, int M) {
    if (K < 32 || K % 32 || N < 32 || N % 32 || M < 1 || M > kMaxRows) return -1;
    const int C = padded_k(K) / 64;
    return (int64_t)(kScratchHeader + (size_t)(N / 32 * 4 + 255) / 256 * 256 + gemm_scratch_floats(C, N) * 4);
}

int dfl_q41_gemm(const void *img, int K, int N, const void *act, int M, float *y, void *scratch, size_t scratch_bytes,
                 void *stream) {
    const int64_t need = dfl_q41_gemm_scratch_bytes(K, N, M);
    if (need < 0 || !img || !act || !y || !scratch || (int64_t)scratch_bytes < need) return DFL_E_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(scratch) & 255) return DFL_E_INVALID_ARG;
    const int C = padded_k(K) / 64;
    GemmArgs a{};
    a.img = static_cast<const uint8_t *>(img);
    a.K = K;
    a.C = C;
    a.N = N;
    a.M = M;
    a.xf = static_cast<const uint32_t *>(act);
    a.xs = reinterpret_cast<const float *>(static_cast<const uint32_t *>(act) + act_words(K));
    a.y = y;
    a.ldy = N;
    a.maxseg = gemm_maxseg(C, N);
    uint8_t *base = static_cast<uint8_t *>(scratch);
    const size_t cbytes = (size_t)(N / 32 * 4 + 255) / 256 * 256;
    a.err = reinterpret_cast<int *>(base);
    a.cnt = reinterpret_cast<int *>(base + kScratchHeader);
    a.part = reinterpret_cast<float *>(base + kScratchHeader + cbytes);
    return launch_gemm(W_Q41, EPI_F32, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFL_OK : DFL_E_CUDA;
}

int dfl_q41_gemm_status(const void *scratch, void *stream) {
    if (!scratch) return DFL_E_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int err = 0;
    if (cudaMemcpyAsync(&err, scratch, sizeof err, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DFL_E_CUDA;
    if (!(err & kErrWaitTimeout)) return DFL_OK;
    if (cudaMemsetAsync(const_cast<void *>(scratch), 0, sizeof err, s) != cudaSuccess) return DFL_E_CUDA;
    return DFL_E_TIMEOUT;
}

// ---- the bf16 head on its own ------------------------------------------------------------------------
int64_t dfl_bf16_image_bytes(int K, int N) {
    if (K < 64 || K % 64 || N < 16 || N % 16) return -1;
    return (int64_t)bf16_image_bytes(K, N);
}

int dfl_bf16_pack(const void *src, int K, int N, void *img, void *stream) {
    if (!src || !img || dfl_bf16_image_bytes(K, N) < 0) return DFL_E_INVALID_ARG;
    return launch_pack_bf16(static_cast<const uint16_t *>(src), K, N, static_cast<uint8_t *>(img),
                            static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFL_OK : DFL_E_CUDA;
}

// scratch: the CTA arrival counter (256-byte header), then per-CTA maxima and their indices
int64_t dfl_bf16_head_scratch_bytes(int K, int N, int M) {
    if (dfl_bf16_image_bytes(K, N) < 0 || M < 1 || M > kMaxRows) return -1;
    return (int64_t)(kScratchHeader + (size_t)head_grid(K / 64, M, N) * kMaxRows * 8);
}

int dfl_bf16_head_argmax(const void *img, int K, int N, const void *act, int M, int32_t *argmax, float *logits,
                         void *scratch, size_t scratch_bytes, void *stream) {
    const int64_t need = dfl_bf16_head_scratch_bytes(K, N, M);
    if (need < 0 || !img || !act || !argmax || !scratch || (int64_t)scratch_bytes < need) return DFL_E_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(scratch) & 255) return DFL_E_INVALID_ARG;
    const int C = K / 64, G = head_grid(C, M, N);
    uint8_t *base = static_cast<uint8_t *>(scratch);
    GemmArgs a{};
    a.img = static_cast<const uint8_t *>(img);
    a.K = K;
    a.C = C;
    a.N = N;
    a.M = M;
    a.xf = static_cast<const uint32_t *>(act);
    a.xs = reinterpret_cast<const float *>(static_cast<const uint32_t *>(act) + act_words(K));
    a.logits = logits;
    a.ldl = N;
    a.am_cnt = reinterpret_cast<int *>(base);
    a.am_val = reinterpret_cast<float *>(base + kScratchHeader);
    a.am_idx = reinterpret_cast<int *>(base + kScratchHeader + (size_t)G * kMaxRows * 4);
    a.am_dst = AM_OUT;
    a.am_out = argmax;
    return launch_gemm(W_BF16, EPI_ARGMAX, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DFL_OK : DFL_E_CUDA;
}

// ---- the product with library-owned scratch -------------------------------------------------------
// One static device array holds the error word, arrival counters and segment partials of
// dfl_q41_gemm_noalloc; its address is looked up once per device and cached (dropped again by
// dfl_q41_gemm_noalloc_reset).
}  // extern "C"

namespace {
constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];
constexpr int kNoallocDevices = kMaxDevices;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoallocDevices] = {};

// this device's copy of the array (the device must be current); nullptr on failure
void *noalloc_scratch() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        // the current device is `dev`: the address is this device's copy of the array
        if (cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_noalloc_scratch) != cudaSuccess) {
            g_noalloc_ptr[dev] = nullptr;
            return nullptr;
        }
    }
    return g_noalloc_ptr[dev];
}
}  // namespace

extern "C" {

int64_t dfl_q41_gemm_noalloc_max_scratch(void) { return (int64_t)kNoallocScratchBytes; }

int dfl_q41_gemm_noalloc(const void *img, int K, int N, const void *act, int M, float *y, void *stream) {
    const int64_t need = dfl_q41_gemm_scratch_bytes(K, N, M);
    if (need < 0 || !img || !act || !y) return DFL_E_INVALID_ARG;
    if ((size_t)need > kNoallocScratchBytes) return DFL_E_CAPACITY;
    void *scratch = noalloc_scratch();
    if (!scratch) return DFL_E_CUDA;
    return dfl_q41_gemm(img, K, N, act, M, y, scratch, kNoallocScratchBytes, stream);
}

int dfl_q41_gemm_noalloc_status(void *stream) {
    void *scratch = noalloc_scratch();
    if (!scratch) return DFL_E_CUDA;
    return dfl_q41_gemm_status(scratch, stream);
}

int dfl_q41_gemm_noalloc_reset(void *stream) {
    const int dev = current_device();
    if (dev < 0) return DFL_E_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        g_noalloc_ptr[dev] = nullptr;   // looked up again: the context may have been recreated
    }
    void *scratch = noalloc_scratch();
    if (!scratch) return DFL_E_CUDA;
    return cudaMemsetAsync(scratch, 0, kNoallocScratchBytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DFL_OK : DFL_E_CUDA;
}

}  // extern "C"
