// Host side of the C ABI declared in include/mk.h: argument checks, TMA
// descriptor encoding, RoPE table, workspace ownership and the launch.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "mk_internal.h"


struct mk_state {
    mk_model_desc desc;
    bool f32 = false;                   // all-fp32 model: the FFMA kernel build
    int device = 0, grid = 0;
    size_t smem = 0;
    // device allocations
    DModel *d_model = nullptr;
    DLayer *d_layers = nullptr;
    CUtensorMap *d_maps = nullptr;      // weight descriptors
    CUtensorMap *d_kvmaps = nullptr;    // [L][2]
    void **d_kpool = nullptr, **d_vpool = nullptr;
    float *d_kvscale = nullptr;         // [L][2] (K, V) scales of an FP8 cache
    std::vector<void *> allocs;
    Ctrl *ctrl = nullptr;
    // KV binding cache
    std::vector<void *> bound_k, bound_v;
    std::vector<float> bound_scale;
    int bound_pages = -1;
    // host-buffer entry point staging
    int32_t *d_tok = nullptr, *d_pos = nullptr, *d_acc = nullptr, *d_am = nullptr;
    float *d_logits = nullptr;
    cudaStream_t last_stream = nullptr;
    int32_t *trace = nullptr;
    float *wtrace = nullptr;
    unsigned long long *stage_trace = nullptr;
    int stage_cap = 0;
    unsigned long long *marks = nullptr;
    int skip_barrier = 0;
    bool launched = false;
    char err[512] = {0};
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};

namespace {

thread_local char g_create_err[512];

mk_status fail(mk_state *st, mk_status s, const char *fmt, ...) {
    if (st) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(st->err, sizeof(st->err), fmt, ap);
        va_end(ap);
    }
    return s;
}

#define CK(call)                                                                        \
    do {                                                                                \
        cudaError_t e_ = (call);                                                        \
        if (e_ != cudaSuccess) return fail(st, MK_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

template <class T>
mk_status dalloc(mk_state *st, T **p, size_t bytes) {
    void *q = nullptr;
    if (cudaMalloc(&q, bytes ? bytes : 16) != cudaSuccess) {
        cudaGetLastError();
        return fail(st, MK_ERR_NOMEM, "cudaMalloc of %zu bytes failed", bytes);
    }
    st->allocs.push_back(q);
    *p = reinterpret_cast<T *>(q);
    return MK_OK;
}

int dt_size(int dt) { return dt == MK_DT_F32 ? 4 : dt == MK_DT_BF16 ? 2 : 1; }

CUtensorMapDataType dt_map(int es) {
    return es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                   : es == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// 2-D [rows][cols] or 3-D [E][rows][cols] tensor, 128-byte x box_rows boxes, 128B swizzle
mk_status encode_map(mk_state *st, CUtensorMap *out, const void *base, int es, long long cols,
                     long long rows, long long E, int box_rows) {
    if (!base) return fail(st, MK_ERR_INVALID, "null weight pointer");
    if (reinterpret_cast<uintptr_t>(base) % 16) return fail(st, MK_ERR_INVALID, "weight pointer not 16-byte aligned");
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)(cols * es), (cuuint64_t)(cols * rows * es)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    cuuint32_t rank = E > 1 ? 3 : 2;
    CUresult r = st->encode(out, dt_map(es), rank, const_cast<void *>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(st, MK_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return MK_OK;
}

// E8M0 scales of an MXFP4 matrix or expert stack, bytes [E][groups][rows]
// (groups = cols/32): boxes of 256 rows x the 8 groups of one 256-column tile
mk_status encode_scale_map(mk_state *st, CUtensorMap *out, const void *base, long long rows, long long groups,
                           long long E) {
    if (!base) return fail(st, MK_ERR_INVALID, "MXFP4 matrix without scales");
    if (reinterpret_cast<uintptr_t>(base) % 16 || rows % 16)
        return fail(st, MK_ERR_INVALID, "MXFP4 scales need a 16-byte aligned pointer and rows % 16 == 0");
    cuuint64_t dims[3] = {(cuuint64_t)rows, (cuuint64_t)groups, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)rows, (cuuint64_t)(rows * groups)};
    cuuint32_t box[3] = {256, 8, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    cuuint32_t rank = E > 1 ? 3 : 2;
    CUresult r = st->encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void *>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(st, MK_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (%d)", (int)r);
    return MK_OK;
}

struct MatSpec {
    const void *w;
    const void *scale;
    int dtype, rows, cols, E;
};

// A matrix descriptor's fields and its tensor maps: tm[0] for the codes and,
// for MXFP4, tm[1] for the E8M0 scales (*nmaps says how many).  The map
// pointers of d are left null; the caller points them at device copies.
mk_status describe_mat(mk_state *st, DMat &d, const MatSpec &s, CUtensorMap *tm, int *nmaps) {
    memset(&d, 0, sizeof(d));
    *nmaps = 0;
    if (!s.w) return MK_OK;  // absent (shared expert with n_shared = 0)
    const bool fp4 = s.dtype == MK_DT_MXFP4_B32;
    d.dtype = s.dtype;
    d.rows = s.rows;
    d.cols = s.cols;
    d.es = dt_size(s.dtype);
    d.cpk = fp4 ? 256 : 128 / d.es;
    d.n_rg = (s.rows + 255) / 256;
    d.n_kc = s.cols / d.cpk;
    d.is3d = s.E > 1;
    d.scale = reinterpret_cast<const float *>(s.scale);
    d.scale_estride = (long long)(s.cols / 128) * s.rows;
    if (s.dtype == MK_DT_FP8E4M3_B128) {
        if (!s.scale) return fail(st, MK_ERR_INVALID, "FP8 matrix without scales");
        if (reinterpret_cast<uintptr_t>(s.scale) % 16) return fail(st, MK_ERR_INVALID, "scale pointer not 16-byte aligned");
    }
    mk_status r = encode_map(st, &tm[0], s.w, d.es, fp4 ? s.cols / 2 : s.cols, s.rows, s.E, 256);
    if (r != MK_OK) return r;
    *nmaps = 1;
    if (fp4) {
        if ((r = encode_scale_map(st, &tm[1], s.scale, s.rows, s.cols / 32, s.E)) != MK_OK) return r;
        *nmaps = 2;
    }
    return MK_OK;
}

// describe_mat for mk_create: maps are appended to `maps` and d's map pointers
// hold (index + 1) until the maps have a device copy
mk_status make_mat(mk_state *st, std::vector<CUtensorMap> &maps, DMat &d, const MatSpec &s) {
    CUtensorMap tm[2];
    int n = 0;
    mk_status r = describe_mat(st, d, s, tm, &n);
    if (r != MK_OK) return r;
    if (n >= 1) {
        d.tmap = reinterpret_cast<const CUtensorMap *>((uintptr_t)(maps.size() + 1));
        maps.push_back(tm[0]);
    }
    if (n == 2) {
        d.smap = reinterpret_cast<const CUtensorMap *>((uintptr_t)(maps.size() + 1));
        maps.push_back(tm[1]);
    }
    return MK_OK;
}

mk_status check_desc(mk_state *st, const mk_model_desc *d) {
    if (d->version != MK_DESC_VERSION) return fail(st, MK_ERR_INVALID, "desc version %d != %d", d->version, MK_DESC_VERSION);
    if (d->n_layers < 1 || d->hidden <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->n_experts <= 0 ||
        d->top_k <= 0 || d->expert_inter <= 0 || d->max_T < 1 || d->max_pages_per_stream < 1)
        return fail(st, MK_ERR_INVALID, "non-positive dimension in desc");
    if (d->max_T > MK_MAXT) return fail(st, MK_ERR_UNSUPPORTED, "max_T %d > %d", d->max_T, MK_MAXT);
    if (d->hidden % 128 || d->hidden > 128 * MK_MAXKB) return fail(st, MK_ERR_UNSUPPORTED, "hidden must be a multiple of 128 and <= 4096");
    if ((d->n_q_heads * d->head_dim) % 128 || d->n_q_heads * d->head_dim > 128 * MK_MAXKB)
        return fail(st, MK_ERR_UNSUPPORTED, "n_q_heads*head_dim must be a multiple of 128 and <= 4096");
    if (d->expert_inter % 128 || d->expert_inter > 128 * MK_MAXKB) return fail(st, MK_ERR_UNSUPPORTED, "expert_inter must be a multiple of 128 and <= 4096");
    if (d->head_dim != 64 && d->head_dim != 128) return fail(st, MK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (d->n_q_heads % d->n_kv_heads) return fail(st, MK_ERR_INVALID, "n_q_heads not a multiple of n_kv_heads");
    if (d->page_size != 64) return fail(st, MK_ERR_UNSUPPORTED, "page_size must be 64");
    if (d->n_experts > MK_MAXE || d->n_experts % 4) return fail(st, MK_ERR_UNSUPPORTED, "n_experts must be a multiple of 4 and <= 512");
    if (d->top_k > MK_MAXK || d->top_k > d->n_experts) return fail(st, MK_ERR_UNSUPPORTED, "top_k must be <= 8 and <= n_experts");
    if (d->n_shared != 0 && d->n_shared != 1) return fail(st, MK_ERR_UNSUPPORTED, "n_shared must be 0 or 1");
    int G = d->n_q_heads / d->n_kv_heads;
    if (G * d->max_T > MK_MAXROWS) return fail(st, MK_ERR_UNSUPPORTED, "(n_q_heads/n_kv_heads)*max_T > 64");
    if (d->kv_dtype != MK_DT_F32 && d->kv_dtype != MK_DT_BF16 && d->kv_dtype != MK_DT_FP8E4M3)
        return fail(st, MK_ERR_UNSUPPORTED, "kv_dtype must be F32, BF16 or FP8E4M3");
    // all-fp32 models run the FFMA kernel (attention over head_dim 64, f32 or
    // bf16 KV); bf16 / FP8 models run the tensor-core kernel (head_dim 128, bf16 KV)
    if (d->weight_dtype == MK_DT_F32) {
        if (d->head_dim != 64) return fail(st, MK_ERR_UNSUPPORTED, "fp32 weights need head_dim 64");
        if (G * d->max_T > 16) return fail(st, MK_ERR_UNSUPPORTED, "fp32 weights support (n_q_heads/n_kv_heads)*T <= 16");
    } else if ((d->kv_dtype != MK_DT_BF16 && d->kv_dtype != MK_DT_FP8E4M3) || d->head_dim != 128) {
        return fail(st, MK_ERR_UNSUPPORTED, "bf16 / FP8 weights need a bf16 or FP8 KV cache and head_dim 128");
    }
    if (d->weight_dtype < 0 || d->weight_dtype > 2) return fail(st, MK_ERR_UNSUPPORTED, "weight_dtype");
    if ((d->weight_dtype == MK_DT_F32) != (d->router_dtype == MK_DT_F32))
        return fail(st, MK_ERR_UNSUPPORTED, "router_dtype must be F32 exactly when weight_dtype is F32");
    if (d->router_dtype != MK_DT_F32 && d->router_dtype != MK_DT_BF16) return fail(st, MK_ERR_UNSUPPORTED, "router_dtype must be F32 or BF16");
    if (d->weight_dtype == MK_DT_F32 &&
        (d->hidden > 2048 || d->n_q_heads * d->head_dim > 2048 || d->expert_inter > 2048))
        return fail(st, MK_ERR_UNSUPPORTED, "F32 weights need hidden, n_q_heads*head_dim, expert_inter <= 2048");
    if (d->vocab < 0) return fail(st, MK_ERR_INVALID, "vocab < 0");
    if (d->lm_head_dtype != MK_DT_BF16 && d->lm_head_dtype != MK_DT_FP8E4M3_B128)
        return fail(st, MK_ERR_UNSUPPORTED, "lm_head_dtype must be BF16 or FP8E4M3_B128");
    if (d->lm_head_dtype == MK_DT_FP8E4M3_B128 && d->weight_dtype == MK_DT_F32)
        return fail(st, MK_ERR_UNSUPPORTED, "an FP8 LM head needs bf16 or FP8 weights elsewhere");
    if (d->expert_dtype != d->weight_dtype) {
        if (d->expert_dtype != MK_DT_MXFP4_B32)
            return fail(st, MK_ERR_UNSUPPORTED, "expert_dtype must equal weight_dtype or be MXFP4");
        if (d->weight_dtype == MK_DT_F32) return fail(st, MK_ERR_UNSUPPORTED, "MXFP4 experts need bf16 or FP8 weights elsewhere");
        if (d->hidden % 256 || d->expert_inter % 256)
            return fail(st, MK_ERR_UNSUPPORTED, "MXFP4 experts need hidden and expert_inter multiples of 256");
    }
    return MK_OK;
}

}  // namespace

extern "C" {

const char *mk_status_string(mk_status s) {
    switch (s) {
        case MK_OK: return "ok";
        case MK_ERR_INVALID: return "invalid argument";
        case MK_ERR_UNSUPPORTED: return "unsupported configuration";
        case MK_ERR_NOMEM: return "out of device memory";
        case MK_ERR_TIMEOUT: return "device-side wait timed out";
        case MK_ERR_CUDA: return "CUDA runtime error";
        case MK_ERR_BAD_STATE: return "bad state";
        case MK_ERR_BAD_INPUT: return "device-side input check failed";
        case MK_ERR_RANGE: return "value outside the kernel's number range";
    }
    return "unknown status";
}

const char *mk_last_error(const mk_state *st) { return st ? st->err : g_create_err; }

void mk_destroy(mk_state *st) {
    if (!st) return;
    cudaDeviceSynchronize();
    for (void *p : st->allocs) cudaFree(p);
    delete st;
}

mk_status mk_create(const mk_model_desc *desc, const mk_weights *w, mk_state **out) {
    if (!desc || !w || !out) return MK_ERR_INVALID;
    *out = nullptr;
    mk_state *st = new mk_state();
    st->desc = *desc;
    mk_status r = check_desc(st, desc);
    auto bail = [&](mk_status s) {
        // keep the message, free the rest
        snprintf(g_create_err, sizeof(g_create_err), "%s", st->err);
        mk_destroy(st);
        return s;
    };
    if (r != MK_OK) return bail(r);
    mk_model_desc &d = st->desc;
    if (d.timeout_ms <= 0) d.timeout_ms = 1000;
    if (!w->layers) return bail(fail(st, MK_ERR_INVALID, "weights.layers is null"));
    if (d.vocab > 0 && (!w->embed || !w->lm_head || !w->final_norm))
        return bail(fail(st, MK_ERR_INVALID, "vocab > 0 needs embed, final_norm and lm_head"));

    // device checks: sm_103 and a co-resident persistent grid, no fallback
    if (cudaGetDevice(&st->device) != cudaSuccess) return bail(fail(st, MK_ERR_CUDA, "no CUDA device"));
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, st->device) != cudaSuccess) return bail(fail(st, MK_ERR_CUDA, "cudaGetDeviceProperties"));
    if (prop.major != 10 || prop.minor != 3)
        return bail(fail(st, MK_ERR_UNSUPPORTED, "built for compute capability 10.3, device is %d.%d", prop.major, prop.minor));
    if (!prop.cooperativeLaunch) return bail(fail(st, MK_ERR_UNSUPPORTED, "device lacks cooperative launch"));
    st->smem = SM_TOTAL + 1024;
    if (st->smem > (size_t)prop.sharedMemPerBlockOptin)
        return bail(fail(st, MK_ERR_UNSUPPORTED, "needs %zu bytes of shared memory per block", st->smem));
    st->f32 = d.weight_dtype == MK_DT_F32;
    if (mk_kernel_setup(st->smem, st->f32) != cudaSuccess) return bail(fail(st, MK_ERR_CUDA, "cudaFuncSetAttribute"));
    int per_sm = mk_kernel_max_blocks(st->smem, st->f32);
    if (per_sm < 1) return bail(fail(st, MK_ERR_UNSUPPORTED, "persistent CTA does not fit on an SM"));
    st->grid = prop.multiProcessorCount;  // one persistent CTA per SM

    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return bail(fail(st, MK_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled not available"));
    st->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);

    const int L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads, hd = d.head_dim;
    const int E = d.n_experts, I = d.expert_inter, nqkv = (Hq + 2 * Hkv) * hd;
    // descriptors of every weight matrix
    std::vector<CUtensorMap> maps;
    std::vector<DLayer> layers(L);
    for (int l = 0; l < L; ++l) {
        const mk_layer_weights &lw = w->layers[l];
        DLayer &dl = layers[l];
        if (!lw.attn_norm || !lw.moe_norm || !lw.router_bias)
            return bail(fail(st, MK_ERR_INVALID, "layer %d: null norm or bias", l));
        if (d.n_shared && (!lw.ws1 || !lw.ws3 || !lw.ws2))
            return bail(fail(st, MK_ERR_INVALID, "layer %d: n_shared = 1 needs ws1/ws3/ws2", l));
        dl.attn_norm = lw.attn_norm;
        dl.moe_norm = lw.moe_norm;
        dl.router_bias = lw.router_bias;
        int wd = d.weight_dtype;
        MatSpec specs[9] = {
            {lw.w_qkv, lw.w_qkv_scale, wd, nqkv, H, 1},
            {lw.w_o, lw.w_o_scale, wd, H, Hq * hd, 1},
            {lw.w_router, nullptr, d.router_dtype, E, H, 1},
            {lw.w1, lw.w1_scale, d.expert_dtype, I, H, E},
            {lw.w3, lw.w3_scale, d.expert_dtype, I, H, E},
            {lw.w2, lw.w2_scale, d.expert_dtype, H, I, E},
            {d.n_shared ? lw.ws1 : nullptr, lw.ws1_scale, wd, I, H, 1},
            {d.n_shared ? lw.ws3 : nullptr, lw.ws3_scale, wd, I, H, 1},
            {d.n_shared ? lw.ws2 : nullptr, lw.ws2_scale, wd, H, I, 1},
        };
        DMat *dm[9] = {&dl.qkv, &dl.o, &dl.router, &dl.w1, &dl.w3, &dl.w2, &dl.s1, &dl.s3, &dl.s2};
        for (int k = 0; k < 9; ++k) {
            if (k < 6 && !specs[k].w) return bail(fail(st, MK_ERR_INVALID, "layer %d: null weight %d", l, k));
            r = make_mat(st, maps, *dm[k], specs[k]);
            if (r != MK_OK) return bail(r);
        }
    }
    DModel hm;
    memset(&hm, 0, sizeof(hm));
    if (d.vocab > 0) {
        MatSpec s{w->lm_head, w->lm_head_scale, d.lm_head_dtype, d.vocab, H, 1};
        r = make_mat(st, maps, hm.lm, s);
        if (r != MK_OK) return bail(r);
    }
    if ((r = dalloc(st, &st->d_maps, maps.size() * sizeof(CUtensorMap))) != MK_OK) return bail(r);
    if (cudaMemcpy(st->d_maps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess)
        return bail(fail(st, MK_ERR_CUDA, "copy of tensor maps"));
    auto fix = [&](DMat &m) {
        if (m.tmap) m.tmap = st->d_maps + ((uintptr_t)m.tmap - 1);
        if (m.smap) m.smap = st->d_maps + ((uintptr_t)m.smap - 1);
    };
    for (auto &dl : layers) {
        fix(dl.qkv); fix(dl.o); fix(dl.router); fix(dl.w1); fix(dl.w3); fix(dl.w2);
        fix(dl.s1); fix(dl.s3); fix(dl.s2);
    }
    fix(hm.lm);
    if ((r = dalloc(st, &st->d_layers, L * sizeof(DLayer))) != MK_OK) return bail(r);
    if (cudaMemcpy(st->d_layers, layers.data(), L * sizeof(DLayer), cudaMemcpyHostToDevice) != cudaSuccess)
        return bail(fail(st, MK_ERR_CUDA, "copy of layer table"));

    // RoPE table: angles in fp64 on the host, stored as fp32 (cos, sin)
    const long long max_pos = (long long)d.max_pages_per_stream * d.page_size;
    std::vector<float2> rope((size_t)max_pos * (hd / 2));
    for (int i = 0; i < hd / 2; ++i) {
        double inv = std::pow((double)d.rope_base, -2.0 * i / hd);
        for (long long p = 0; p < max_pos; ++p) {
            double a = (double)p * inv;
            rope[(size_t)p * (hd / 2) + i] = make_float2((float)std::cos(a), (float)std::sin(a));
        }
    }
    float2 *d_rope;
    if ((r = dalloc(st, &d_rope, rope.size() * sizeof(float2))) != MK_OK) return bail(r);
    if (cudaMemcpy(d_rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
        return bail(fail(st, MK_ERR_CUDA, "copy of rope table"));

    // workspace
    hm.L = L; hm.H = H; hm.Hq = Hq; hm.Hkv = Hkv; hm.d = hd; hm.E = E; hm.K = d.top_k; hm.I = I;
    hm.V = d.vocab; hm.P = d.page_size; hm.nshared = d.n_shared; hm.max_pages = d.max_pages_per_stream;
    hm.maxT = d.max_T; hm.G = st->grid; hm.wdt = d.weight_dtype; hm.rdt = d.router_dtype;
    hm.kvdt = d.kv_dtype; hm.kv_es = dt_size(d.kv_dtype); hm.nqkv = nqkv; hm.eps = d.rms_eps;
    hm.timeout_ns = (long long)d.timeout_ms * 1000000ll;
    hm.layers = st->d_layers;
    hm.embed = reinterpret_cast<const uint16_t *>(w->embed);
    hm.final_norm = w->final_norm;
    hm.rope = d_rope;
    const size_t T8 = MK_MAXT;
    if ((r = dalloc(st, &st->ctrl, sizeof(Ctrl))) != MK_OK) return bail(r);
    hm.ctrl = st->ctrl;
    if ((r = dalloc(st, &hm.att_cnt, sizeof(int) * L * Hkv)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.o_buf, 4 * T8 * Hq * hd)) != MK_OK) return bail(r);
    if (cudaMemset(hm.att_cnt, 0, sizeof(int) * L * Hkv) != cudaSuccess) return bail(fail(st, MK_ERR_CUDA, "memset"));
    if ((r = dalloc(st, &hm.qkv_acc, 2 * 8 * T8 * nqkv)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.res, 8 * T8 * H)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.rlog, 2 * 8 * T8 * E)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.sh_acc, 2 * 8 * T8 * 2 * I)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.ea_acc, 2 * 8 * T8 * d.top_k * 2 * I)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.logit_acc, 8 * T8 * (d.vocab > 0 ? d.vocab : 1))) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.ssq, 4 * 3 * MK_MAXKB * T8)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.att_part, 4ull * Hkv * MK_MAXSPLIT * MK_MAXROWS * (hd + 2))) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.cand_v, 4 * T8 * st->grid)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.cand_i, 4 * T8 * st->grid)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.cand_m, 4 * T8 * st->grid)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &hm.cand_s, 4 * T8 * st->grid)) != MK_OK) return bail(r);
    if (cudaMemset(st->ctrl, 0, sizeof(Ctrl)) != cudaSuccess) return bail(fail(st, MK_ERR_CUDA, "memset ctrl"));
    if ((r = dalloc(st, &st->d_model, sizeof(DModel))) != MK_OK) return bail(r);
    if (cudaMemcpy(st->d_model, &hm, sizeof(DModel), cudaMemcpyHostToDevice) != cudaSuccess)
        return bail(fail(st, MK_ERR_CUDA, "copy of model block"));
    if ((r = dalloc(st, &st->d_kvmaps, 2 * L * sizeof(CUtensorMap))) != MK_OK) return bail(r);
    if ((r = dalloc(st, &st->d_kpool, L * sizeof(void *))) != MK_OK) return bail(r);
    if ((r = dalloc(st, &st->d_vpool, L * sizeof(void *))) != MK_OK) return bail(r);
    if ((r = dalloc(st, &st->d_kvscale, 2 * L * sizeof(float))) != MK_OK) return bail(r);
    if ((r = dalloc(st, &st->d_tok, 4 * T8)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &st->d_pos, 4 * T8)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &st->d_acc, 16)) != MK_OK) return bail(r);
    if ((r = dalloc(st, &st->d_am, 4 * T8)) != MK_OK) return bail(r);
    if (d.vocab > 0 && (r = dalloc(st, &st->d_logits, 4 * T8 * d.vocab)) != MK_OK) return bail(r);
    *out = st;
    return MK_OK;
}

static mk_status bind_kv(mk_state *st, const mk_kv_cache *kv) {
    const mk_model_desc &d = st->desc;
    const int L = d.n_layers;
    if (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table || kv->n_pages < 1)
        return fail(st, MK_ERR_INVALID, "bad kv cache descriptor");
    // (K, V) scales: those of an FP8 cache (absent: 1), 1 for other caches
    std::vector<float> sc(2 * L, 1.f);
    if (d.kv_dtype == MK_DT_FP8E4M3) {
        for (int l = 0; l < L; ++l) {
            if (kv->k_scale) sc[2 * l] = kv->k_scale[l];
            if (kv->v_scale) sc[2 * l + 1] = kv->v_scale[l];
            if (!(sc[2 * l] > 0.f) || !(sc[2 * l + 1] > 0.f) || !std::isfinite(sc[2 * l]) || !std::isfinite(sc[2 * l + 1]))
                return fail(st, MK_ERR_INVALID, "FP8 KV scales of layer %d must be finite and > 0", l);
        }
    }
    bool same = st->bound_pages == kv->n_pages && (int)st->bound_k.size() == L && st->bound_scale == sc;
    for (int l = 0; same && l < L; ++l) same = st->bound_k[l] == kv->k_pool[l] && st->bound_v[l] == kv->v_pool[l];
    if (same) return MK_OK;
    // the tables below are read by a step still running on the last stream
    if (st->launched && cudaStreamSynchronize(st->last_stream) != cudaSuccess)
        return fail(st, MK_ERR_CUDA, "synchronize before rebinding the KV cache failed");
    const int es = dt_size(d.kv_dtype);
    std::vector<CUtensorMap> maps(2 * L);
    for (int l = 0; l < L; ++l) {
        long long rows = (long long)kv->n_pages * d.n_kv_heads * d.page_size;
        mk_status r = encode_map(st, &maps[2 * l], kv->k_pool[l], es, d.head_dim, rows, 1, d.page_size);
        if (r != MK_OK) return r;
        r = encode_map(st, &maps[2 * l + 1], kv->v_pool[l], es, d.head_dim, rows, 1, d.page_size);
        if (r != MK_OK) return r;
    }
    CK(cudaMemcpy(st->d_kvmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(st->d_kpool, kv->k_pool, L * sizeof(void *), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(st->d_vpool, kv->v_pool, L * sizeof(void *), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(st->d_kvscale, sc.data(), 2 * L * sizeof(float), cudaMemcpyHostToDevice));
    st->bound_scale = sc;
    st->bound_k.assign(kv->k_pool, kv->k_pool + L);
    st->bound_v.assign(kv->v_pool, kv->v_pool + L);
    st->bound_pages = kv->n_pages;
    return MK_OK;
}

static mk_status launch(mk_state *st, Params &p, void *stream) {
    p.m = st->d_model;
    p.stage_trace = st->stage_trace;
    p.stage_cap = st->stage_cap;
    p.marks = st->marks;
    p.skip_barrier = st->skip_barrier;
    p.kvmaps = st->d_kvmaps;
    p.kpool = st->d_kpool;
    p.vpool = st->d_vpool;
    p.kv_scale = st->d_kvscale;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = mk_launch(p, st->grid, st->smem, s, st->f32);
    if (e != cudaSuccess) return fail(st, MK_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    st->last_stream = s;
    st->launched = true;
    return MK_OK;
}

mk_status mk_decode_step(mk_state *st, const int32_t *draft_tokens, int T, const int32_t *positions,
                         const mk_kv_cache *kv, float *out_logits, int32_t *out_accepted,
                         int32_t *out_argmax, void *stream) {
    if (!st) return MK_ERR_INVALID;
    if (st->desc.vocab <= 0) return fail(st, MK_ERR_BAD_STATE, "model has no LM head (vocab = 0)");
    if (T < 1 || T > st->desc.max_T) return fail(st, MK_ERR_INVALID, "T = %d outside [1, %d]", T, st->desc.max_T);
    if (!draft_tokens || !positions || !out_logits || !out_accepted)
        return fail(st, MK_ERR_INVALID, "null pointer argument");
    mk_status r = bind_kv(st, kv);
    if (r != MK_OK) return r;
    Params p;
    memset(&p, 0, sizeof(p));
    p.page_table = kv->page_table;
    p.tokens = draft_tokens;
    p.positions = positions;
    p.T = T;
    p.mode = 0;
    p.n_pages = kv->n_pages;
    p.out_logits = out_logits;
    p.out_accepted = out_accepted;
    p.out_argmax = out_argmax;
    p.trace = st->trace;
    p.wtrace = st->wtrace;
    return launch(st, p, stream);
}

mk_status mk_decode_step_sample(mk_state *st, const int32_t *draft_tokens, int T, const int32_t *positions,
                                const mk_kv_cache *kv, float temperature, const float *uniforms,
                                float *out_logits, int32_t *out_accepted, int32_t *out_token, void *stream) {
    if (!st) return MK_ERR_INVALID;
    if (st->desc.vocab <= 0) return fail(st, MK_ERR_BAD_STATE, "model has no LM head (vocab = 0)");
    if (T < 1 || T > st->desc.max_T) return fail(st, MK_ERR_INVALID, "T = %d outside [1, %d]", T, st->desc.max_T);
    if (!draft_tokens || !positions || !out_logits || !out_accepted || !uniforms || !out_token)
        return fail(st, MK_ERR_INVALID, "null pointer argument");
    if (!(temperature >= 1e-3f && temperature <= 1e3f))
        return fail(st, MK_ERR_INVALID, "temperature must lie in [1e-3, 1e3]");
    mk_status r = bind_kv(st, kv);
    if (r != MK_OK) return r;
    Params p;
    memset(&p, 0, sizeof(p));
    p.page_table = kv->page_table;
    p.tokens = draft_tokens;
    p.positions = positions;
    p.T = T;
    p.mode = 0;
    p.n_pages = kv->n_pages;
    p.out_logits = out_logits;
    p.out_accepted = out_accepted;
    p.temperature = temperature;
    p.uniforms = uniforms;
    p.out_token = out_token;
    p.trace = st->trace;
    p.wtrace = st->wtrace;
    return launch(st, p, stream);
}

mk_status mk_decode_batch(mk_state *st, int n_streams, const int32_t *draft_tokens, int T,
                          const int32_t *positions, const mk_kv_cache *kv, float *out_logits,
                          int32_t *out_accepted, int32_t *out_argmax, void *stream) {
    if (!st) return MK_ERR_INVALID;
    if (n_streams < 1) return fail(st, MK_ERR_INVALID, "n_streams = %d", n_streams);
    if (!kv || !kv->page_table) return fail(st, MK_ERR_INVALID, "bad kv cache descriptor");
    const long long V = st->desc.vocab, P = st->desc.max_pages_per_stream;
    for (int s = 0; s < n_streams; ++s) {
        mk_kv_cache row = *kv;
        row.page_table = kv->page_table + (long long)s * P;
        mk_status r = mk_decode_step(st, draft_tokens ? draft_tokens + (long long)s * T : nullptr, T,
                                     positions ? positions + (long long)s * T : nullptr, &row,
                                     out_logits ? out_logits + (long long)s * T * V : nullptr,
                                     out_accepted ? out_accepted + s : nullptr,
                                     out_argmax ? out_argmax + (long long)s * T : nullptr, stream);
        if (r != MK_OK) return r;
    }
    return MK_OK;
}

mk_status mk_decode_step_host(mk_state *st, const int32_t *h_tokens, int T, const int32_t *h_positions,
                              const mk_kv_cache *kv, float *h_logits, int32_t *h_accepted,
                              int32_t *h_argmax, void *stream) {
    if (!st) return MK_ERR_INVALID;
    if (T < 1 || T > st->desc.max_T) return fail(st, MK_ERR_INVALID, "T = %d outside [1, %d]", T, st->desc.max_T);
    if (!h_tokens || !h_positions || !h_accepted) return fail(st, MK_ERR_INVALID, "null pointer argument");
    if (st->desc.vocab <= 0) return fail(st, MK_ERR_BAD_STATE, "model has no LM head (vocab = 0)");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CK(cudaMemcpyAsync(st->d_tok, h_tokens, 4 * T, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(st->d_pos, h_positions, 4 * T, cudaMemcpyHostToDevice, s));
    mk_status r = mk_decode_step(st, st->d_tok, T, st->d_pos, kv, st->d_logits, st->d_acc, st->d_am, stream);
    if (r != MK_OK) return r;
    if (h_logits) CK(cudaMemcpyAsync(h_logits, st->d_logits, sizeof(float) * T * st->desc.vocab, cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(h_accepted, st->d_acc, 4, cudaMemcpyDeviceToHost, s));
    if (h_argmax) CK(cudaMemcpyAsync(h_argmax, st->d_am, 4 * T, cudaMemcpyDeviceToHost, s));
    return mk_get_status(st);
}

mk_status mk_layer_forward(mk_state *st, int layer, const float *hidden_in, int T, const int32_t *positions,
                           const mk_kv_cache *kv, float *hidden_out, int32_t *out_topk_idx,
                           float *out_topk_w, void *stream) {
    if (!st) return MK_ERR_INVALID;
    if (layer < 0 || layer >= st->desc.n_layers) return fail(st, MK_ERR_INVALID, "layer %d out of range", layer);
    if (T < 1 || T > st->desc.max_T) return fail(st, MK_ERR_INVALID, "T = %d outside [1, %d]", T, st->desc.max_T);
    if (!hidden_in || !hidden_out || !positions) return fail(st, MK_ERR_INVALID, "null pointer argument");
    if (hidden_in == hidden_out) return fail(st, MK_ERR_INVALID, "hidden_in and hidden_out alias");
    mk_status r = bind_kv(st, kv);
    if (r != MK_OK) return r;
    Params p;
    memset(&p, 0, sizeof(p));
    p.page_table = kv->page_table;
    p.positions = positions;
    p.T = T;
    p.mode = 1;
    p.layer = layer;
    p.n_pages = kv->n_pages;
    p.hidden_in = hidden_in;
    p.hidden_out = hidden_out;
    p.out_idx = out_topk_idx;
    p.out_w = out_topk_w;
    return launch(st, p, stream);
}

mk_status mk_set_routing_trace(mk_state *st, int32_t *idx_trace, float *w_trace) {
    if (!st) return MK_ERR_INVALID;
    st->trace = idx_trace;
    st->wtrace = w_trace;
    return MK_OK;
}

mk_status mk_set_stage_trace(mk_state *st, uint64_t *times, int capacity, uint64_t *events) {
    if (!st || (times && capacity < 1)) return MK_ERR_INVALID;
    st->stage_trace = reinterpret_cast<unsigned long long *>(times);
    st->stage_cap = times ? capacity : 0;
    st->marks = reinterpret_cast<unsigned long long *>(events);
    return MK_OK;
}

mk_status mk_debug_skip_barrier(mk_state *st, int barrier) {
    if (!st || barrier < 0) return MK_ERR_INVALID;
    st->skip_barrier = barrier;
    return MK_OK;
}

mk_status mk_get_status(mk_state *st) {
    if (!st) return MK_ERR_INVALID;
    CK(cudaStreamSynchronize(st->last_stream));
    Ctrl c;
    CK(cudaMemcpy(&c, st->ctrl, sizeof(Ctrl), cudaMemcpyDeviceToHost));
    if (c.status != 0) fail(st, (mk_status)c.status, "device status %d at check %d", c.status, c.where);
    return (mk_status)c.status;
}

mk_status mk_get_stats(mk_state *st, mk_stats *out) {
    if (!st || !out) return MK_ERR_INVALID;
    CK(cudaStreamSynchronize(st->last_stream));
    Ctrl c;
    CK(cudaMemcpy(&c, st->ctrl, sizeof(Ctrl), cudaMemcpyDeviceToHost));
    memset(out, 0, sizeof(*out));
    out->steps = c.steps;
    out->accepted_sum = c.accepted_sum;
    out->distinct_experts_sum = c.distinct_sum;
    out->last_accepted = c.last_accepted;
    out->last_distinct_experts = c.last_distinct;
    out->fused = 1;
    out->grid_ctas = st->grid;
    out->launches_per_step = 1;
    out->barriers_per_step = 6 * st->desc.n_layers + 3;
    return MK_OK;
}

mk_status mk_reset(mk_state *st) {
    if (!st) return MK_ERR_INVALID;
    CK(cudaDeviceSynchronize());
    CK(cudaMemset(st->ctrl, 0, sizeof(Ctrl)));
    return MK_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// mk_layer_forward_noalloc: the same kernel in one-layer mode, for callers that
// cannot allocate device memory (an allocator-less runtime, a plugin host that
// owns all device memory, code that must not allocate after start-up).  Calls
// stage their tables with copies from host memory, so they are refused during
// stream capture.  Everything the launch needs besides the
// caller's tensors -- the model block, the layer's TMA descriptors, the RoPE
// rows of the step, the control block and all accumulators -- is carved out of
// one file-scope device array, so no call allocates.
// ---------------------------------------------------------------------------
#define MK_NOALLOC_SCRATCH_BYTES (24u << 20)  // 24 MiB, held by every device that loads the library
static __device__ __align__(256) unsigned char g_mk_noalloc_scratch[MK_NOALLOC_SCRATCH_BYTES];

namespace {
struct NoallocDevice {
    bool ready;
    unsigned char *scratch;   // device address of g_mk_noalloc_scratch on this device
    int grid;
    size_t smem;
    PFN_cuTensorMapEncodeTiled_v12000 encode;
};
constexpr int kMaxDevices = 64;
NoallocDevice g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// per-device set-up, run by the first call on a device with that device current
mk_status noalloc_setup(mk_state *st, int dev, NoallocDevice **out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(st, MK_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocDevice &d = g_noalloc[dev];
    if (!d.ready) {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_mk_noalloc_scratch);
        if (e != cudaSuccess || !ptr) return fail(st, MK_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return fail(st, MK_ERR_CUDA, "cudaGetDeviceProperties");
        if (prop.major != 10 || prop.minor != 3)
            return fail(st, MK_ERR_UNSUPPORTED, "built for compute capability 10.3, device is %d.%d", prop.major, prop.minor);
        const size_t smem = SM_TOTAL + 1024;
        for (int f = 0; f < 2; ++f) {
            if (mk_kernel_setup(smem, f != 0) != cudaSuccess) return fail(st, MK_ERR_CUDA, "cudaFuncSetAttribute");
            if (mk_kernel_max_blocks(smem, f != 0) < 1) return fail(st, MK_ERR_UNSUPPORTED, "persistent CTA does not fit on an SM");
        }
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return fail(st, MK_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled not available");
        d.scratch = static_cast<unsigned char *>(ptr);
        d.grid = prop.multiProcessorCount;
        d.smem = smem;
        d.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        d.ready = true;
    }
    *out = &d;
    return MK_OK;
}

// bump allocator over the static array (offsets only; nothing is allocated)
struct Carve {
    size_t off = 0;
    template <class T>
    size_t take(size_t bytes) {
        size_t o = (off + 255) & ~(size_t)255;
        off = o + (bytes ? bytes : 16);
        return o;
    }
};
}  // namespace

extern "C" mk_status mk_layer_forward_noalloc(const mk_model_desc *desc, const mk_layer_weights *lw,
                                              void *k_pool, void *v_pool, const int32_t *page_table,
                                              int n_pages, const float *hidden_in, int T, int ctx,
                                              const int32_t *positions, float *hidden_out,
                                              int32_t *out_topk_idx, float *out_topk_w,
                                              int32_t *out_status, void *stream) {
    mk_state local;  // carries the error text and the encode entry point; owns nothing
    mk_state *st = &local;
    auto ret = [&](mk_status s) {
        snprintf(g_create_err, sizeof(g_create_err), "%s", st->err);
        return s;
    };
#define CKN(call)                                                                                  \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess) return ret(fail(st, MK_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_))); \
    } while (0)
    if (!desc || !lw || !k_pool || !v_pool || !page_table || !hidden_in || !hidden_out || !positions)
        return ret(fail(st, MK_ERR_INVALID, "null pointer argument"));
    mk_status r = check_desc(st, desc);
    if (r != MK_OK) return ret(r);
    mk_model_desc d = *desc;
    if (d.kv_dtype == MK_DT_FP8E4M3)
        return ret(fail(st, MK_ERR_UNSUPPORTED, "mk_layer_forward_noalloc takes no KV scales: FP8 caches are not supported"));
    if (T < 1 || T > d.max_T) return ret(fail(st, MK_ERR_INVALID, "T = %d outside [1, %d]", T, d.max_T));
    if (ctx < 0 || (long long)ctx + T > (long long)d.max_pages_per_stream * d.page_size)
        return ret(fail(st, MK_ERR_INVALID, "ctx %d + T exceeds the page table", ctx));
    if (n_pages < 1) return ret(fail(st, MK_ERR_INVALID, "n_pages < 1"));
    if (hidden_in == hidden_out) return ret(fail(st, MK_ERR_INVALID, "hidden_in and hidden_out alias"));
    if (d.timeout_ms <= 0) d.timeout_ms = 1000;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ret(fail(st, MK_ERR_CUDA, "no CUDA device"));
    {
        // the tables below are staged with copies from this call's stack: a
        // captured graph would replay them from memory that no longer holds them
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs) != cudaSuccess)
            return ret(fail(st, MK_ERR_CUDA, "cudaStreamIsCapturing failed"));
        if (cs != cudaStreamCaptureStatusNone)
            return ret(fail(st, MK_ERR_UNSUPPORTED, "mk_layer_forward_noalloc cannot be called during stream capture"));
    }
    NoallocDevice *nd = nullptr;
    if ((r = noalloc_setup(st, dev, &nd)) != MK_OK) return ret(r);
    st->encode = nd->encode;

    const int H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads, hd = d.head_dim;
    const int E = d.n_experts, I = d.expert_inter, nqkv = (Hq + 2 * Hkv) * hd;
    const size_t T8 = MK_MAXT;
    // layout of the static array for this model
    Carve cv;
    const size_t o_model = cv.take<DModel>(sizeof(DModel));
    const size_t o_layer = cv.take<DLayer>(sizeof(DLayer));
    const size_t o_maps = cv.take<CUtensorMap>(14 * sizeof(CUtensorMap));
    const size_t o_pools = cv.take<void *>(2 * sizeof(void *));
    const size_t o_rope = cv.take<float2>(T8 * (hd / 2) * sizeof(float2));
    const size_t o_ctrl = cv.take<Ctrl>(sizeof(Ctrl));
    const size_t o_attcnt = cv.take<int>(sizeof(int) * Hkv);
    const size_t o_obuf = cv.take<float>(4 * T8 * Hq * hd);
    const size_t o_qkv = cv.take<long long>(2 * 8 * T8 * nqkv);
    const size_t o_res = cv.take<long long>(8 * T8 * H);
    const size_t o_rlog = cv.take<long long>(2 * 8 * T8 * E);
    const size_t o_sh = cv.take<long long>(2 * 8 * T8 * 2 * I);
    const size_t o_ea = cv.take<long long>(2 * 8 * T8 * d.top_k * 2 * I);
    const size_t o_logit = cv.take<long long>(8 * T8);
    const size_t o_ssq = cv.take<float>(4 * 3 * MK_MAXKB * T8);
    const size_t o_part = cv.take<float>(4ull * Hkv * MK_MAXSPLIT * MK_MAXROWS * (hd + 2));
    const size_t o_candv = cv.take<float>(4 * T8 * nd->grid);
    const size_t o_candi = cv.take<int>(4 * T8 * nd->grid);
    const size_t o_candm = cv.take<float>(4 * T8 * nd->grid);
    const size_t o_cands = cv.take<float>(4 * T8 * nd->grid);
    if (cv.off > MK_NOALLOC_SCRATCH_BYTES)
        return ret(fail(st, MK_ERR_UNSUPPORTED, "model needs %zu bytes of scratch; mk_layer_forward_noalloc has %u",
                        cv.off, (unsigned)MK_NOALLOC_SCRATCH_BYTES));
    unsigned char *base = nd->scratch;

    // descriptors of the layer's matrices and of its KV pools
    // 9 matrices with up to 3 MXFP4 scale maps, then the K and V pools
    constexpr int kMatMaps = 12;
    CUtensorMap maps[kMatMaps + 2];
    DLayer dl;
    memset(&dl, 0, sizeof(dl));
    dl.attn_norm = lw->attn_norm;
    dl.moe_norm = lw->moe_norm;
    dl.router_bias = lw->router_bias;
    if (!lw->attn_norm || !lw->moe_norm || !lw->router_bias) return ret(fail(st, MK_ERR_INVALID, "null norm or bias"));
    if (d.n_shared && (!lw->ws1 || !lw->ws3 || !lw->ws2)) return ret(fail(st, MK_ERR_INVALID, "n_shared = 1 needs ws1/ws3/ws2"));
    const int wd = d.weight_dtype, xd = d.expert_dtype;
    MatSpec specs[9] = {
        {lw->w_qkv, lw->w_qkv_scale, wd, nqkv, H, 1},   {lw->w_o, lw->w_o_scale, wd, H, Hq * hd, 1},
        {lw->w_router, nullptr, d.router_dtype, E, H, 1}, {lw->w1, lw->w1_scale, xd, I, H, E},
        {lw->w3, lw->w3_scale, xd, I, H, E},             {lw->w2, lw->w2_scale, xd, H, I, E},
        {d.n_shared ? lw->ws1 : nullptr, lw->ws1_scale, wd, I, H, 1},
        {d.n_shared ? lw->ws3 : nullptr, lw->ws3_scale, wd, I, H, 1},
        {d.n_shared ? lw->ws2 : nullptr, lw->ws2_scale, wd, H, I, 1},
    };
    DMat *dm[9] = {&dl.qkv, &dl.o, &dl.router, &dl.w1, &dl.w3, &dl.w2, &dl.s1, &dl.s3, &dl.s2};
    int nmaps = 0;
    for (int k = 0; k < 9; ++k) {
        if (k < 6 && !specs[k].w) return ret(fail(st, MK_ERR_INVALID, "null weight %d", k));
        int n = 0;
        if ((r = describe_mat(st, *dm[k], specs[k], &maps[nmaps], &n)) != MK_OK) return ret(r);
        if (n >= 1) dm[k]->tmap = reinterpret_cast<const CUtensorMap *>(base + o_maps) + nmaps;
        if (n == 2) dm[k]->smap = reinterpret_cast<const CUtensorMap *>(base + o_maps) + nmaps + 1;
        nmaps += n;
    }
    const int kv_es = dt_size(d.kv_dtype);
    const long long kv_rows = (long long)n_pages * Hkv * d.page_size;
    if ((r = encode_map(st, &maps[kMatMaps], k_pool, kv_es, hd, kv_rows, 1, d.page_size)) != MK_OK) return ret(r);
    if ((r = encode_map(st, &maps[kMatMaps + 1], v_pool, kv_es, hd, kv_rows, 1, d.page_size)) != MK_OK) return ret(r);

    // RoPE rows of positions ctx..ctx+T-1 (fp64 angles, stored fp32); the model
    // block points the table so that the kernel's absolute index lands on them
    float2 rope[MK_MAXT * 64];
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < hd / 2; ++i) {
            double a = (double)(ctx + t) * std::pow((double)d.rope_base, -2.0 * i / hd);
            rope[t * (hd / 2) + i] = make_float2((float)std::cos(a), (float)std::sin(a));
        }

    DModel hm;
    memset(&hm, 0, sizeof(hm));
    hm.L = 1; hm.H = H; hm.Hq = Hq; hm.Hkv = Hkv; hm.d = hd; hm.E = E; hm.K = d.top_k; hm.I = I;
    hm.V = 0; hm.P = d.page_size; hm.nshared = d.n_shared; hm.max_pages = d.max_pages_per_stream;
    hm.maxT = d.max_T; hm.G = nd->grid; hm.wdt = d.weight_dtype; hm.rdt = d.router_dtype;
    hm.kvdt = d.kv_dtype; hm.kv_es = kv_es; hm.nqkv = nqkv; hm.eps = d.rms_eps;
    hm.timeout_ns = (long long)d.timeout_ms * 1000000ll;
    hm.layers = reinterpret_cast<const DLayer *>(base + o_layer);
    hm.rope = reinterpret_cast<const float2 *>(base + o_rope) - (long long)ctx * (hd / 2);
    hm.ctrl = reinterpret_cast<Ctrl *>(base + o_ctrl);
    hm.att_cnt = reinterpret_cast<int *>(base + o_attcnt);
    hm.o_buf = reinterpret_cast<float *>(base + o_obuf);
    hm.qkv_acc = reinterpret_cast<long long *>(base + o_qkv);
    hm.res = reinterpret_cast<long long *>(base + o_res);
    hm.rlog = reinterpret_cast<long long *>(base + o_rlog);
    hm.sh_acc = reinterpret_cast<long long *>(base + o_sh);
    hm.ea_acc = reinterpret_cast<long long *>(base + o_ea);
    hm.logit_acc = reinterpret_cast<long long *>(base + o_logit);
    hm.ssq = reinterpret_cast<float *>(base + o_ssq);
    hm.att_part = reinterpret_cast<float *>(base + o_part);
    hm.cand_v = reinterpret_cast<float *>(base + o_candv);
    hm.cand_i = reinterpret_cast<int *>(base + o_candi);
    hm.cand_m = reinterpret_cast<float *>(base + o_candm);
    hm.cand_s = reinterpret_cast<float *>(base + o_cands);
    void *pools[2] = {k_pool, v_pool};

    // stage the launch's tables into the array (stream-ordered copies; the host
    // buffers may be reused once the calls return) and clear the control block
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CKN(cudaMemcpyAsync(base + o_model, &hm, sizeof(hm), cudaMemcpyHostToDevice, s));
    CKN(cudaMemcpyAsync(base + o_layer, &dl, sizeof(dl), cudaMemcpyHostToDevice, s));
    CKN(cudaMemcpyAsync(base + o_maps, maps, sizeof(maps), cudaMemcpyHostToDevice, s));
    CKN(cudaMemcpyAsync(base + o_pools, pools, sizeof(pools), cudaMemcpyHostToDevice, s));
    CKN(cudaMemcpyAsync(base + o_rope, rope, sizeof(float2) * T * (hd / 2), cudaMemcpyHostToDevice, s));
    CKN(cudaMemsetAsync(base + o_ctrl, 0, sizeof(Ctrl), s));

    Params p;
    memset(&p, 0, sizeof(p));
    p.m = reinterpret_cast<const DModel *>(base + o_model);
    p.kvmaps = reinterpret_cast<const CUtensorMap *>(base + o_maps) + kMatMaps;
    p.kpool = reinterpret_cast<void *const *>(base + o_pools);
    p.vpool = reinterpret_cast<void *const *>(base + o_pools) + 1;
    p.page_table = page_table;
    p.positions = positions;
    p.T = T;
    p.mode = 1;
    p.layer = 0;
    p.n_pages = n_pages;
    p.hidden_in = hidden_in;
    p.hidden_out = hidden_out;
    p.out_idx = out_topk_idx;
    p.out_w = out_topk_w;
    p.host_ctx1 = ctx + 1;  // the RoPE rows above exist for positions ctx .. ctx+T-1 only
    cudaError_t e = mk_launch(p, nd->grid, nd->smem, s, d.weight_dtype == MK_DT_F32);
    if (e != cudaSuccess) return ret(fail(st, MK_ERR_CUDA, "launch: %s", cudaGetErrorString(e)));
    if (out_status)
        CKN(cudaMemcpyAsync(out_status, base + o_ctrl + offsetof(Ctrl, status), sizeof(int32_t),
                           cudaMemcpyDeviceToDevice, s));
    return MK_OK;
#undef CKN
}
