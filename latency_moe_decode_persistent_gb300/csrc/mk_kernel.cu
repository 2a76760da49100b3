// Persistent verify-step megakernel for sm_103a.
//
// One cooperative launch runs a whole speculative-verify step: embedding, every
// decoder layer (RMSNorm + QKV GEMV + RoPE + KV append + split-K GQA attention,
// O projection + residual, router GEMV + sigmoid + bitonic top-k, routed and
// shared SwiGLU experts + residual), the final norm, the LM head, argmax and the
// accept-prefix count.  This replaces the ~1,300 small kernels per step that the
// single-GB300 decode analysis ("Why one GB300 doesn't beat 4x RTX PRO 6000 at
// single-stream decode", section "Where the 11.2 ms goes") counts, and keeps one
// persistent CTA per SM as the megakernel plugin does ("DeepSeek-V4.1-Flash breaks
// 1,000 tokens per second for one user", section "What NVIDIA shipped").
//
// Structure of a CTA (288 threads):
//   warp 8      producer: walks the CTA's static chunk schedule for the whole
//               step and streams weight tiles / KV pages into an 8-slot shared
//               memory ring with TMA (cp.async.bulk.tensor, 128-byte swizzle)
//               plus 1-D bulk copies of FP8 block scales.  It runs ahead across
//               grid barriers; it only stops for a free slot, and for the router
//               result before the routed-expert tiles of a layer.
//   warps 0..7  consumers: every 16 KB tile is 128 rows x 128 bytes of one
//               matrix; warp w reduces rows 16w..16w+15 against the T <= 8
//               activations with mma.sync m16n8k16 (tokens are the N=8 side;
//               FP8 codes are widened to f16 in registers, scales applied per
//               1x128 block), accumulating across consecutive tiles of a row
//               group, then adds its partial into a global fixed-point (2^-32)
//               int64 accumulator.  Integer adds make every cross-CTA reduction
//               order-independent, so the step is bitwise deterministic.
// RMSNorm is folded: GEMVs consume gamma*x and the consumer of their result
// divides by rms(x), whose sum of squares is computed by 32 CTAs in parallel.
// Grid barriers (monotonic counter, acquire/release) separate the stages; every
// wait is bounded by %globaltimer and turns into a status code.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "mk_internal.h"

namespace {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t sa(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(tx)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(sa(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *map, int x, int y,
                                      uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(sa(dst)),
        "l"(map), "r"(x), "r"(y), "r"(sa(bar))
        : "memory");
}
__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                      uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sa(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(sa(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(sa(dst)),
        "l"(src), "r"(bytes), "r"(sa(bar))
        : "memory");
}
__device__ __forceinline__ void bar_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(MK_NCWARPS * 32) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                      uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                       uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void mma_f16(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// two FP8 E4M3 codes (low byte first) -> f16x2 (low half first)
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t v16) {
    uint32_t r;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
        : "=r"(r)
        : "r"(v16));
    return r;
}
// two bf16 (low half first) -> f16x2
__device__ __forceinline__ uint32_t bf16x2_f16x2(uint32_t v) {
    float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ long long to_fx(float v) { return __float2ll_rn(v * MK_FX); }
__device__ __forceinline__ float from_fx(long long v) {
    return __ll2float_rn(v) * (1.0f / MK_FX);
}
__device__ __forceinline__ void red_add(long long *p, long long v) {
    atomicAdd(reinterpret_cast<unsigned long long *>(p), (unsigned long long)v);
}
__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// byte address of (row, byte) inside a TMA box stored with the 128-byte swizzle
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int byte) {
    return base + row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
}

// ------------------------------------------------------------------ CTA context
struct RouteSm {
    int nd;
    int dlist[MK_MAXD];
    signed char dslot[MK_MAXD][MK_MAXT];
    int idx[MK_MAXT][MK_MAXK];
    float w[MK_MAXT][MK_MAXK];
};
struct MiscSm {
    int abort;
    int gs_ok;
    int emask[16];
    float inv_rms[3][MK_MAXT];   // attention, moe, final
    int distinct_total;
    int valid, ctx;
    int pad;
    unsigned long long base;
};

struct Ctx {
    const Params *p;
    const DModel *m;
    Ctrl *ctrl;
    unsigned char *sm;
    uint64_t *full, *empty, *route;
    RouteSm *rt;          // [2]
    MiscSm *misc;
    int cta, G, T, ctx, nsplit, tid, warp, lane;
    unsigned long long bar_base;
    int nbar;
    long long timeout;
};

__device__ __forceinline__ bool aborted(const Ctx &c) {
    return *(volatile int *)&c.misc->abort != 0 || *(volatile int *)&c.ctrl->abort != 0;
}
__device__ void raise_err(const Ctx &c, int code, int where) {
    *(volatile int *)&c.misc->abort = 1;
    if (atomicCAS(&c.ctrl->status, 0, code) == 0) atomicExch(&c.ctrl->where, where);
    atomicExch(&c.ctrl->abort, 1);
}
// bounded wait on an mbarrier phase
__device__ bool mbar_wait(uint64_t *b, uint32_t parity, const Ctx &c, int where) {
    if (mbar_try(b, parity)) return true;
    uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(b, parity)) return true;
        if ((it & 15) == 0) {
            if (aborted(c)) return false;
            if ((long long)(gtimer() - t0) > c.timeout) {
                raise_err(c, MK_ERR_TIMEOUT, where);
                return false;
            }
        }
    }
}
// bounded wait that ignores the abort flag (drain of copies in flight)
__device__ void mbar_wait_drain(uint64_t *b, uint32_t parity, const Ctx &c) {
    uint64_t t0 = gtimer();
    while (!mbar_try(b, parity)) {
        if ((long long)(gtimer() - t0) > c.timeout) return;
    }
}
__device__ bool spin_ge_u64(unsigned long long *a, unsigned long long target, const Ctx &c,
                            int where) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
        if (v >= target) return true;
        if ((it & 31) == 31) {
            if (aborted(c)) return false;
            uint64_t now = gtimer();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > c.timeout) {
                raise_err(c, MK_ERR_TIMEOUT, where);
                return false;
            }
        }
    }
}
__device__ bool spin_ge_s32(int *a, int target, const Ctx &c, int where) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
        if (v >= target) return true;
        if ((it & 31) == 31) {
            if (aborted(c)) return false;
            uint64_t now = gtimer();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > c.timeout) {
                raise_err(c, MK_ERR_TIMEOUT, where);
                return false;
            }
        }
    }
}

// grid-wide barrier among the consumer warps of all CTAs; split into arrive/wait
__device__ void grid_arrive(Ctx &c) {
    bar_consumers();
    c.nbar++;
    if (c.tid == 0) {
        __threadfence();
        atomicAdd(&c.ctrl->bar_count, 1ull);
    }
}
__device__ bool grid_wait(Ctx &c, int where) {
    if (c.tid == 0) {
        bool ok = !aborted(c);
        if (ok) ok = spin_ge_u64(&c.ctrl->bar_count, c.bar_base + (unsigned long long)c.nbar * c.G, c,
                                 where);
        __threadfence();
        c.misc->gs_ok = ok && !aborted(c);
    }
    bar_consumers();
    return c.misc->gs_ok != 0;
}
__device__ bool grid_sync(Ctx &c, int where) {
    grid_arrive(c);
    return grid_wait(c, where);
}

// ------------------------------------------------------------------ schedules
struct Item {
    const DMat *m;
    int e, rg, kc, mat, ex;
};

__device__ __forceinline__ void split_range(int total, int parts, int part, int &b, int &e) {
    b = (int)((long long)total * part / parts);
    e = (int)((long long)total * (part + 1) / parts);
}

__device__ int stage_total(const DModel &m, int st, const DLayer &L, const RouteSm *rt) {
    switch (st) {
        case ST_QKV: return L.qkv.n_rg * L.qkv.n_kc;
        case ST_O: return L.o.n_rg * L.o.n_kc;
        case ST_ROUTER: return L.router.n_rg * L.router.n_kc;
        case ST_SHA: return m.nshared ? 2 * L.s1.n_rg * L.s1.n_kc : 0;
        case ST_EXPA: return rt->nd * 2 * L.w1.n_rg * L.w1.n_kc;
        case ST_EXPB: return (rt->nd + m.nshared) * L.w2.n_rg * L.w2.n_kc;
        case ST_LM: return m.lm.n_rg * m.lm.n_kc;
    }
    return 0;
}

__device__ Item stage_item(const DModel &m, int st, const DLayer &L, const RouteSm *rt, int idx) {
    Item it;
    it.e = 0;
    it.mat = 0;
    it.ex = 0;
    const DMat *d;
    int r = idx;
    switch (st) {
        case ST_QKV: d = &L.qkv; break;
        case ST_O: d = &L.o; break;
        case ST_ROUTER: d = &L.router; break;
        case ST_LM: d = &m.lm; break;
        case ST_SHA: {
            int per = L.s1.n_rg * L.s1.n_kc;
            it.mat = r / per;
            r -= it.mat * per;
            d = it.mat ? &L.s3 : &L.s1;
            break;
        }
        case ST_EXPA: {
            int per1 = L.w1.n_rg * L.w1.n_kc;
            it.ex = r / (2 * per1);
            r -= it.ex * 2 * per1;
            it.mat = r / per1;
            r -= it.mat * per1;
            d = it.mat ? &L.w3 : &L.w1;
            it.e = rt->dlist[it.ex];
            break;
        }
        default: {  // ST_EXPB
            int per = L.w2.n_rg * L.w2.n_kc;
            it.ex = r / per;
            r -= it.ex * per;
            if (it.ex < rt->nd) {
                d = &L.w2;
                it.e = rt->dlist[it.ex];
            } else {
                d = &L.s2;
            }
            break;
        }
    }
    it.m = d;
    it.rg = r / d->n_kc;
    it.kc = r - it.rg * d->n_kc;
    return it;
}

// attention split of a unit (one kv head, a run of pages)
struct AttUnit {
    bool active, has_new;
    int g, s, p0, pc1;
};
__device__ AttUnit att_unit(const Ctx &c) {
    const DModel &m = *c.m;
    AttUnit u;
    int ncp = (c.ctx + m.P - 1) / m.P, np = ncp + 1;
    u.active = c.cta < m.Hkv * c.nsplit;
    u.g = c.cta / c.nsplit;
    u.s = c.cta - u.g * c.nsplit;
    int p1;
    split_range(np, c.nsplit, u.s, u.p0, p1);
    u.pc1 = min(p1, ncp);
    u.has_new = (p1 == np);
    return u;
}

// ------------------------------------------------------------------ producer
__device__ bool prod_slot(Ctx &c, uint32_t &pi, uint32_t bytes, uint32_t &slot) {
    slot = pi % MK_RING;
    if (!mbar_wait(&c.empty[slot], ((pi / MK_RING) & 1) ^ 1, c, 100)) return false;
    mbar_expect_tx(&c.full[slot], bytes);
    return true;
}

__device__ bool prod_gemv(Ctx &c, int st, const DLayer &L, const RouteSm *rt, uint32_t &pi) {
    const DModel &m = *c.m;
    int b, e;
    split_range(stage_total(m, st, L, rt), c.G, c.cta, b, e);
    for (int idx = b; idx < e; ++idx) {
        Item it = stage_item(m, st, L, rt, idx);
        const DMat &d = *it.m;
        uint32_t sbytes = 0;
        if (d.dtype == MK_DT_FP8E4M3_B128) sbytes = min(128, d.rows - it.rg * 128) * 4;
        uint32_t slot;
        if (!prod_slot(c, pi, MK_SLOT + sbytes, slot)) return false;
        void *dst = c.sm + SM_RING + slot * MK_SLOT;
        int x = it.kc * (128 / d.es);
        if (d.is3d) tma3d(dst, d.tmap, x, it.rg * 128, it.e, &c.full[slot]);
        else tma2d(dst, d.tmap, x, it.rg * 128, &c.full[slot]);
        if (sbytes) {
            const float *src = d.scale + (long long)it.e * d.scale_estride +
                               (long long)it.kc * d.rows + it.rg * 128;
            bulk_g2s(c.sm + SM_SCALE + slot * 512, src, sbytes, &c.full[slot]);
        }
        ++pi;
    }
    return true;
}

__device__ bool prod_att(Ctx &c, int l, uint32_t &pi) {
    const DModel &m = *c.m;
    AttUnit u = att_unit(c);
    if (!u.active) return true;
    int nbox = (m.d * m.kv_es) / 128;
    const CUtensorMap *km = c.p->kvmaps + 2 * l, *vm = km + 1;
    for (int j = u.p0; j < u.pc1; ++j) {
        int phys = __ldg(c.p->page_table + j);
        int y = (phys * m.Hkv + u.g) * m.P;
        for (int kv = 0; kv < 2; ++kv) {
            uint32_t slot;
            if (!prod_slot(c, pi, nbox * m.P * 128, slot)) return false;
            unsigned char *dst = c.sm + SM_RING + slot * MK_SLOT;
            for (int bx = 0; bx < nbox; ++bx)
                tma2d(dst + bx * m.P * 128, kv ? vm : km, bx * (128 / m.kv_es), y, &c.full[slot]);
            ++pi;
        }
    }
    return true;
}

__device__ void producer(Ctx &c) {
    const DModel &m = *c.m;
    const Params &p = *c.p;
    uint32_t pi = 0;
    int nl = p.mode ? 1 : m.L;
    bool ok = true;
    for (int li = 0; li < nl && ok; ++li) {
        int l = p.mode ? p.layer : li;
        const DLayer &L = m.layers[l];
        const RouteSm *rt = &c.rt[li & 1];
        ok = prod_gemv(c, ST_QKV, L, rt, pi) && prod_att(c, l, pi) &&
             prod_gemv(c, ST_O, L, rt, pi) && prod_gemv(c, ST_ROUTER, L, rt, pi) &&
             prod_gemv(c, ST_SHA, L, rt, pi);
        if (!ok) break;
        if (!mbar_wait(c.route, li & 1, c, 101)) { ok = false; break; }
        ok = prod_gemv(c, ST_EXPA, L, rt, pi) && prod_gemv(c, ST_EXPB, L, rt, pi);
    }
    if (ok && p.mode == 0) ok = prod_gemv(c, ST_LM, m.layers[0], &c.rt[0], pi);
    if (!ok) {
        // copies still in flight must land before the CTA may exit
        for (uint32_t i = (pi > MK_RING ? pi - MK_RING : 0); i < pi; ++i)
            mbar_wait_drain(&c.full[i % MK_RING], (i / MK_RING) & 1, c);
    }
}

// ------------------------------------------------------------------ activations
// Fragment order of the B operand (activations) of one 128-column block: for
// step s (0..7) and lane l = 4n + q the lane holds token n's columns
//   32q + 8*(((s>>1) + 2*(q>>1)) & 3) + 4*(s&1) + j,  j = 0..3,
// as two f16x2 words.  The weight side reads the same columns (a permutation of
// the reduction index shared by both operands), which lets every lane fetch its
// FP8/bf16 weights as whole 16-byte swizzled chunks without bank conflicts.
__device__ __forceinline__ int frag_col(int s, int q, int j) {
    return 32 * q + 8 * (((s >> 1) + 2 * (q >> 1)) & 3) + 4 * (s & 1) + j;
}

// source of a GEMV input: fixed-point [T][stride] times gamma, or float [T][stride]
struct ActSrc {
    const long long *fx;
    const float *f32;
    int stride;
    const float *gamma;
};
__device__ __forceinline__ float act_val(const ActSrc &a, int t, int col) {
    float v = a.fx ? from_fx(__ldcg(a.fx + (long long)t * a.stride + col))
                   : __ldcg(a.f32 + (long long)t * a.stride + col);
    return a.gamma ? v * __ldg(a.gamma + col) : v;
}

// build f16 fragments for the 128-column blocks in `mask` (consumer threads)
__device__ void build_frags(const Ctx &c, const ActSrc &a, uint32_t mask, int kb0 = 0) {
    unsigned char *fr = c.sm + SM_SCRATCH;
    const int s = c.tid >> 5, l = c.lane, n = l >> 2, q = l & 3;
    for (int kb = 0; kb < MK_MAXKB; ++kb) {
        if (!((mask >> kb) & 1)) continue;
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = (n < c.T) ? act_val(a, n, (kb + kb0) * 128 + frag_col(s, q, j)) : 0.f;
        uint2 w = make_uint2(pack_f16(v[0], v[1]), pack_f16(v[2], v[3]));
        *reinterpret_cast<uint2 *>(fr + kb * 2048 + ((s >> 1) * 32 + l) * 16 + (s & 1) * 8) = w;
    }
}
// f32 activations [MK_MAXT][K] for the FFMA path
__device__ void build_act32(const Ctx &c, const ActSrc &a, int K) {
    float *dst = reinterpret_cast<float *>(c.sm + SM_SCRATCH);
    for (int i = c.tid; i < MK_MAXT * K; i += MK_NCWARPS * 32) {
        int t = i / K, col = i - t * K;
        dst[i] = t < c.T ? act_val(a, t, col) : 0.f;
    }
}

// k-blocks of a contiguous item range [b, e) over (.., rg, kc) ordered items
__device__ uint32_t needed_kb(int b, int e, const DMat &d) {
    if (e - b >= d.n_kc) return 0xffffffffu >> (32 - (d.cols / 128));
    uint32_t mask = 0;
    for (int i = b; i < e; ++i) {
        int kc = i % d.n_kc;
        mask |= 1u << ((kc * (128 / d.es)) / 128);
    }
    return mask;
}

// ------------------------------------------------------------------ GEMV tiles
struct Tgt {
    long long *base;
    int toff[MK_MAXT];
    float tw[MK_MAXT];
    int row_limit;
};

__device__ void make_tgt(const Ctx &c, int st, const Item &it, const RouteSm *rt, Tgt &g) {
    const DModel &m = *c.m;
    for (int t = 0; t < MK_MAXT; ++t) {
        g.toff[t] = -1;
        g.tw[t] = 1.f;
    }
    g.row_limit = it.m->rows;
    switch (st) {
        case ST_QKV:
            g.base = m.qkv_acc;
            for (int t = 0; t < c.T; ++t) g.toff[t] = t * m.nqkv;
            break;
        case ST_O:
            g.base = m.res;
            for (int t = 0; t < c.T; ++t) g.toff[t] = t * m.H;
            break;
        case ST_ROUTER:
            g.base = m.rlog;
            for (int t = 0; t < c.T; ++t) g.toff[t] = t * m.E;
            break;
        case ST_SHA:
            g.base = m.sh_acc + it.mat * m.I;
            for (int t = 0; t < c.T; ++t) g.toff[t] = t * 2 * m.I;
            break;
        case ST_EXPA:
            g.base = m.ea_acc + it.mat * m.I;
            for (int t = 0; t < c.T; ++t) {
                int j = rt->dslot[it.ex][t];
                if (j >= 0) g.toff[t] = (t * m.K + j) * 2 * m.I;
            }
            break;
        case ST_EXPB:
            g.base = m.res;
            for (int t = 0; t < c.T; ++t) {
                if (it.ex < rt->nd) {
                    int j = rt->dslot[it.ex][t];
                    if (j >= 0) {
                        g.toff[t] = t * m.H;
                        g.tw[t] = rt->w[t][j];
                    }
                } else {
                    g.toff[t] = t * m.H;
                }
            }
            break;
        case ST_LM:
            g.base = m.logit_acc;
            for (int t = 0; t < c.T; ++t) g.toff[t] = t * m.V;
            break;
    }
}

// MMA layout: lane holds rows (r, r+8) x tokens (2q, 2q+1) of the warp's 16 rows
__device__ void flush_mma(const Ctx &c, const Tgt &g, int row0, const float *acc) {
    const int r = c.lane >> 2, q = c.lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int t = 2 * q + (i & 1);
        int row = row0 + r + (i >> 1) * 8;
        if (t < MK_MAXT && g.toff[t] >= 0 && row < g.row_limit)
            red_add(g.base + g.toff[t] + row, to_fx(acc[i] * g.tw[t]));
    }
}
// FFMA layout: lanes 0..15 hold one row each, all tokens
__device__ void flush_f32(const Ctx &c, const Tgt &g, int row0, float *acc) {
    // lanes l and l+16 hold the two column halves of the same row
#pragma unroll
    for (int t = 0; t < MK_MAXT; ++t) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 16);
    if (c.lane >= 16) return;
    int row = row0 + c.lane;
    if (row >= g.row_limit) return;
#pragma unroll
    for (int t = 0; t < MK_MAXT; ++t)
        if (g.toff[t] >= 0) red_add(g.base + g.toff[t] + row, to_fx(acc[t] * g.tw[t]));
}

// one 128-row x 128-byte tile of FP8 or bf16 weights against the f16 fragments
__device__ __forceinline__ void tile_mma(const Ctx &c, const DMat &d, int slot, int kc,
                                         float *acc) {
    const int r = c.lane >> 2, q = c.lane & 3;
    const uint32_t tile = sa(c.sm + SM_RING + slot * MK_SLOT);
    const int row0 = c.warp * 16 + r, row8 = row0 + 8;
    const uint32_t frag = sa(c.sm + SM_SCRATCH);
    if (d.dtype == MK_DT_FP8E4M3_B128) {
        const int ca = 2 * q + (q >> 1), cb = 2 * q + 1 - (q >> 1);
        uint4 a0 = lds128(tile + row0 * 128 + ((ca ^ r) << 4));
        uint4 a1 = lds128(tile + row0 * 128 + ((cb ^ r) << 4));
        uint4 b0 = lds128(tile + row8 * 128 + ((ca ^ r) << 4));
        uint4 b1 = lds128(tile + row8 * 128 + ((cb ^ r) << 4));
        const uint32_t fb = frag + kc * 2048 + c.lane * 16;
        uint4 f0 = lds128(fb), f1 = lds128(fb + 512), f2 = lds128(fb + 1024), f3 = lds128(fb + 1536);
        float k4[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t w0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t w8[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const uint32_t fx[8] = {f0.x, f0.z, f1.x, f1.z, f2.x, f2.z, f3.x, f3.z};
        const uint32_t fy[8] = {f0.y, f0.w, f1.y, f1.w, f2.y, f2.w, f3.y, f3.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            mma_f16(k4, e4m3x2_f16x2(w0[s] & 0xffff), e4m3x2_f16x2(w8[s] & 0xffff),
                    e4m3x2_f16x2(w0[s] >> 16), e4m3x2_f16x2(w8[s] >> 16), fx[s], fy[s]);
        }
        const float *sc = reinterpret_cast<const float *>(c.sm + SM_SCALE + slot * 512);
        float s0 = sc[row0], s8 = sc[row8];
        acc[0] += k4[0] * s0;
        acc[1] += k4[1] * s0;
        acc[2] += k4[2] * s8;
        acc[3] += k4[3] * s8;
    } else {  // bf16: the tile is half of a 128-column block
        const int h = kc & 1, kb = kc >> 1;
        const bool act = (q >> 1) == h;
        const int qq = q & 1;
        uint4 ra[4], rb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int ch = 4 * qq + ((i + 2 * h) & 3);
            if (act) {
                ra[i] = lds128(tile + row0 * 128 + ((ch ^ r) << 4));
                rb[i] = lds128(tile + row8 * 128 + ((ch ^ r) << 4));
            } else {
                ra[i] = make_uint4(0, 0, 0, 0);
                rb[i] = make_uint4(0, 0, 0, 0);
            }
        }
        const uint32_t fb = frag + kb * 2048 + c.lane * 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 f = lds128(fb + i * 512);
            mma_f16(acc, bf16x2_f16x2(ra[i].x), bf16x2_f16x2(rb[i].x), bf16x2_f16x2(ra[i].y),
                    bf16x2_f16x2(rb[i].y), f.x, f.y);
            mma_f16(acc, bf16x2_f16x2(ra[i].z), bf16x2_f16x2(rb[i].z), bf16x2_f16x2(ra[i].w),
                    bf16x2_f16x2(rb[i].w), f.z, f.w);
        }
    }
}

// one 128-row x 32-column fp32 tile with FFMA (tiny fp32 models)
__device__ __forceinline__ void tile_f32(const Ctx &c, const DMat &d, int slot, int kc,
                                         float *acc) {
    const uint32_t tile = sa(c.sm + SM_RING + slot * MK_SLOT);
    const float *act = reinterpret_cast<const float *>(c.sm + SM_SCRATCH);
    const int row = c.warp * 16 + (c.lane & 15), hf = c.lane >> 4;
    const int K = d.cols;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 w = lds128(tile + row * 128 + (((4 * hf + i) ^ (row & 7)) << 4));
        float wv[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                       __uint_as_float(w.w)};
        int col = kc * 32 + 16 * hf + 4 * i;
#pragma unroll
        for (int t = 0; t < MK_MAXT; ++t) {
            if (t < c.T) {
                const float *x = act + t * K + col;
                acc[t] += wv[0] * x[0] + wv[1] * x[1] + wv[2] * x[2] + wv[3] * x[3];
            }
        }
    }
}

// h_e = silu(a/rms) * (b/rms) fragments of one expert (or the shared one)
__device__ void build_h_frags(const Ctx &c, const RouteSm *rt, int ex, bool f32path) {
    const DModel &m = *c.m;
    const bool shared = ex >= rt->nd;
    auto hval = [&](int t, int col) -> float {
        const long long *pa;
        if (shared) {
            pa = m.sh_acc + (long long)t * 2 * m.I;
        } else {
            int j = rt->dslot[ex][t];
            if (j < 0) return 0.f;
            pa = m.ea_acc + (long long)(t * m.K + j) * 2 * m.I;
        }
        float inv = c.misc->inv_rms[1][t];
        float av = from_fx(__ldcg(pa + col)) * inv, bv = from_fx(__ldcg(pa + m.I + col)) * inv;
        return av / (1.f + expf(-av)) * bv;
    };
    if (f32path) {
        float *dst = reinterpret_cast<float *>(c.sm + SM_SCRATCH);
        for (int i = c.tid; i < MK_MAXT * m.I; i += MK_NCWARPS * 32) {
            int t = i / m.I, col = i - t * m.I;
            dst[i] = t < c.T ? hval(t, col) : 0.f;
        }
        return;
    }
    unsigned char *fr = c.sm + SM_SCRATCH;
    const int s = c.tid >> 5, l = c.lane, n = l >> 2, q = l & 3;
    for (int kb = 0; kb < m.I / 128; ++kb) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = n < c.T ? hval(n, kb * 128 + frag_col(s, q, j)) : 0.f;
        *reinterpret_cast<uint2 *>(fr + kb * 2048 + ((s >> 1) * 32 + l) * 16 + (s & 1) * 8) =
            make_uint2(pack_f16(v[0], v[1]), pack_f16(v[2], v[3]));
    }
}

// consume this CTA's tiles of one GEMV stage
__device__ void cons_gemv(Ctx &c, int st, const DLayer &L, const RouteSm *rt, uint32_t &ci) {
    const DModel &m = *c.m;
    int b, e;
    split_range(stage_total(m, st, L, rt), c.G, c.cta, b, e);
    float acc[MK_MAXT];
    const DMat *cm = nullptr;
    int ce = -1, crg = -1, cex = -1, cmat = 0, last_hex = -1;
    Item cur;
    for (int idx = b; idx < e; ++idx) {
        Item it = stage_item(m, st, L, rt, idx);
        const bool f32 = it.m->dtype == MK_DT_F32;
        if (it.m != cm || it.e != ce || it.rg != crg || it.ex != cex || it.mat != cmat) {
            if (cm) {
                Tgt g;
                make_tgt(c, st, cur, rt, g);
                if (cm->dtype == MK_DT_F32) flush_f32(c, g, cur.rg * 128 + c.warp * 16, acc);
                else flush_mma(c, g, cur.rg * 128 + c.warp * 16, acc);
            }
#pragma unroll
            for (int i = 0; i < MK_MAXT; ++i) acc[i] = 0.f;
            cm = it.m;
            ce = it.e;
            crg = it.rg;
            cex = it.ex;
            cmat = it.mat;
            cur = it;
            if (st == ST_EXPB && it.ex != last_hex) {
                bar_consumers();
                build_h_frags(c, rt, it.ex, f32);
                bar_consumers();
                last_hex = it.ex;
            }
        }
        const int slot = ci % MK_RING;
        if (mbar_wait(&c.full[slot], (ci / MK_RING) & 1, c, 200 + st)) {
            if (f32) tile_f32(c, *it.m, slot, it.kc, acc);
            else tile_mma(c, *it.m, slot, it.kc, acc);
        }
        __syncwarp();
        if (c.lane == 0) mbar_arrive(&c.empty[slot]);
        ++ci;
    }
    if (cm) {
        Tgt g;
        make_tgt(c, st, cur, rt, g);
        if (cm->dtype == MK_DT_F32) flush_f32(c, g, cur.rg * 128 + c.warp * 16, acc);
        else flush_mma(c, g, cur.rg * 128 + c.warp * 16, acc);
    }
}

// ------------------------------------------------------------------ small helpers
__device__ void zero_slice(const Ctx &c, long long *p, long long n) {
    long long b = n * c.cta / c.G, e = n * (c.cta + 1) / c.G;
    for (long long i = b + c.tid; i < e; i += MK_NCWARPS * 32) __stcg(p + i, 0ll);
}
// sum of squares of 128-column block `kb` of the residual for every token
__device__ void ssq_block(const Ctx &c, int which) {
    const DModel &m = *c.m;
    int kb = c.cta;
    if (kb >= m.H / 128) return;
    if (c.warp >= c.T) return;
    int t = c.warp;
    float s = 0.f;
    for (int i = c.lane; i < 128; i += 32) {
        float v = from_fx(__ldcg(m.res + (long long)t * m.H + kb * 128 + i));
        s += v * v;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (c.lane == 0) __stcg(m.ssq + (which * MK_MAXKB + kb) * MK_MAXT + t, s);
}
__device__ void compute_inv_rms(const Ctx &c, int which) {
    const DModel &m = *c.m;
    if (c.tid < c.T) {
        float s = 0.f;
        for (int kb = 0; kb < m.H / 128; ++kb) s += __ldcg(m.ssq + (which * MK_MAXKB + kb) * MK_MAXT + c.tid);
        c.misc->inv_rms[which][c.tid] = rsqrtf(s / (float)m.H + m.eps);
    }
}

// ------------------------------------------------------------------ routing
__device__ __forceinline__ unsigned long long key64(float key, int e) {
    uint32_t b = __float_as_uint(key);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)b << 32) | (0xffffffffu - (uint32_t)e);
}
// sort 16 keys descending (bitonic network, registers)
__device__ __forceinline__ void bitonic16_desc(unsigned long long *v) {
#pragma unroll
    for (int k = 2; k <= 16; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                int l = i ^ j;
                if (l > i) {
                    bool desc = (i & k) == 0;
                    unsigned long long a = v[i], b = v[l];
                    bool sw = desc ? (a < b) : (a > b);
                    v[i] = sw ? b : a;
                    v[l] = sw ? a : b;
                }
            }
        }
    }
}

// top-K of each token's sigmoid scores + bias; weights from the unbiased scores
__device__ void route_layer(Ctx &c, const DLayer &L, RouteSm *rt) {
    const DModel &m = *c.m;
    if (c.warp < c.T) {
        const int t = c.warp;
        const float inv = c.misc->inv_rms[1][t];
        unsigned long long v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            int e = c.lane + 32 * i;
            v[i] = 0ull;
            if (e < m.E) {
                float lg = from_fx(__ldcg(m.rlog + (long long)t * m.E + e)) * inv;
                float s = 1.f / (1.f + expf(-lg));
                v[i] = key64(s + __ldg(L.router_bias + e), e);
            }
        }
        bitonic16_desc(v);
        // bitonic merge of the lanes' sorted top-8 lists
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned long long pv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pv[i] = __shfl_xor_sync(0xffffffffu, v[i], o);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = v[i] > pv[7 - i] ? v[i] : pv[7 - i];
#pragma unroll
            for (int j = 4; j > 0; j >>= 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if ((i & j) == 0) {
                        unsigned long long a = v[i], b = v[i + j];
                        v[i] = a > b ? a : b;
                        v[i + j] = a > b ? b : a;
                    }
                }
            }
        }
        // lanes 0..K-1 take entry `lane`
        unsigned long long mine = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i == c.lane) mine = v[i];
        int e = (int)(0xffffffffu - (uint32_t)(mine & 0xffffffffu));
        float s = 0.f;
        if (c.lane < m.K) {
            float lg = from_fx(__ldcg(m.rlog + (long long)t * m.E + e)) * inv;
            s = 1.f / (1.f + expf(-lg));
        }
        float sum = s;
#pragma unroll
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (c.lane < m.K) {
            rt->idx[t][c.lane] = e;
            rt->w[t][c.lane] = s / sum;
        }
    }
    if (c.tid < 16) c.misc->emask[c.tid] = 0;
    bar_consumers();
    if (c.warp == 0) {
        for (int i = c.lane; i < c.T * m.K; i += 32) {
            int e = rt->idx[i / m.K][i % m.K];
            atomicOr(&c.misc->emask[e >> 5], 1 << (e & 31));
        }
        __syncwarp();
        int cnt = c.lane < 16 ? __popc(c.misc->emask[c.lane]) : 0;
        int pre = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, pre, o);
            if (c.lane >= o) pre += y;
        }
        int total = __shfl_sync(0xffffffffu, pre, 31);
        if (c.lane < 16) {
            int pos = pre - cnt;
            uint32_t w = c.misc->emask[c.lane];
            while (w) {
                int bit = __ffs(w) - 1;
                w &= w - 1;
                rt->dlist[pos++] = c.lane * 32 + bit;
            }
        }
        if (c.lane == 0) rt->nd = total;
        for (int i = c.lane; i < MK_MAXD * MK_MAXT; i += 32) (&rt->dslot[0][0])[i] = -1;
        __syncwarp();
        for (int i = c.lane; i < c.T * m.K; i += 32) {
            int t = i / m.K, j = i % m.K, e = rt->idx[t][j];
            int wd = e >> 5;
            int pos = 0;
            for (int k = 0; k < wd; ++k) pos += __popc(c.misc->emask[k]);
            pos += __popc(c.misc->emask[wd] & ((1u << (e & 31)) - 1));
            rt->dslot[pos][t] = (signed char)j;
        }
    }
    bar_consumers();
}

// ------------------------------------------------------------------ attention
// q rows are ordered (t, head-in-group): row = t * G + hh
__device__ float qkv_val(const Ctx &c, int t, int col) {
    return from_fx(__ldcg(c.m->qkv_acc + (long long)t * c.m->nqkv + col)) * c.misc->inv_rms[0][t];
}

// prepares rotated q (scratch) and, for the unit holding the new block, the
// block's K/V (scratch + cache append)
__device__ void att_prepare(const Ctx &c, int l, const AttUnit &u, bool mma_path) {
    const DModel &m = *c.m;
    const int G = m.Hq / m.Hkv, R = G * c.T, hd = m.d / 2;
    unsigned char *scr = c.sm + SM_SCRATCH;
    // rotated queries
    for (int i = c.tid; i < R * hd; i += MK_NCWARPS * 32) {
        int row = i / hd, k = i - row * hd;
        int t = row / G, h = u.g * G + (row - t * G);
        float x1 = qkv_val(c, t, h * m.d + k), x2 = qkv_val(c, t, h * m.d + k + hd);
        float2 cs = __ldg(m.rope + (long long)(c.ctx + t) * hd + k);
        float y1 = x1 * cs.x - x2 * cs.y, y2 = x2 * cs.x + x1 * cs.y;
        if (mma_path) {
            __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(scr);
            qs[row * 136 + k] = __float2bfloat16_rn(y1);
            qs[row * 136 + k + hd] = __float2bfloat16_rn(y2);
        } else {
            float *qs = reinterpret_cast<float *>(scr);
            qs[row * m.d + k] = y1;
            qs[row * m.d + k + hd] = y2;
        }
    }
    if (mma_path) {  // zero the padding rows of the last m-tile
        __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(scr);
        int R16 = (R + 15) & ~15;
        for (int i = c.tid; i < (R16 - R) * 136; i += MK_NCWARPS * 32) qs[R * 136 + i] = __float2bfloat16_rn(0.f);
    }
    if (!u.has_new) return;
    // block keys / values: mini page after the queries
    unsigned char *mini = scr + 17408;
    if (mma_path) {
        for (int i = c.tid; i < 8192 / 16; i += MK_NCWARPS * 32)
            reinterpret_cast<uint4 *>(mini)[i] = make_uint4(0, 0, 0, 0);
    }
    bar_consumers();
    const int kv_es = m.kv_es;
    for (int i = c.tid; i < c.T * hd; i += MK_NCWARPS * 32) {
        int t = i / hd, k = i - t * hd;
        int kc0 = (m.Hq + u.g) * m.d, vc0 = (m.Hq + m.Hkv + u.g) * m.d;
        float x1 = qkv_val(c, t, kc0 + k), x2 = qkv_val(c, t, kc0 + k + hd);
        float2 cs = __ldg(m.rope + (long long)(c.ctx + t) * hd + k);
        float k1 = x1 * cs.x - x2 * cs.y, k2 = x2 * cs.x + x1 * cs.y;
        float v1 = qkv_val(c, t, vc0 + k), v2 = qkv_val(c, t, vc0 + k + hd);
        int pos = c.ctx + t;
        int phys = __ldg(c.p->page_table + pos / m.P);
        long long off = ((long long)(phys * m.Hkv + u.g) * m.P + (pos % m.P)) * m.d;
        if (kv_es == 2) {
            __nv_bfloat16 kb1 = __float2bfloat16_rn(k1), kb2 = __float2bfloat16_rn(k2);
            __nv_bfloat16 vb1 = __float2bfloat16_rn(v1), vb2 = __float2bfloat16_rn(v2);
            __nv_bfloat16 *kp = reinterpret_cast<__nv_bfloat16 *>(c.p->kpool[l]) + off;
            __nv_bfloat16 *vp = reinterpret_cast<__nv_bfloat16 *>(c.p->vpool[l]) + off;
            kp[k] = kb1;
            kp[k + hd] = kb2;
            vp[k] = vb1;
            vp[k + hd] = vb2;
            if (mma_path) {  // [box][16 keys][128 B] swizzled
                auto put = [&](unsigned char *base, int dd, __nv_bfloat16 v) {
                    int byte = dd * 2;
                    int bx = byte >> 7;
                    *reinterpret_cast<__nv_bfloat16 *>(base + (swz(0, t, byte & 127) + bx * 2048)) = v;
                };
                put(mini, k, kb1);
                put(mini, k + hd, kb2);
                put(mini + 4096, k, vb1);
                put(mini + 4096, k + hd, vb2);
            } else {
                float *mk = reinterpret_cast<float *>(mini);
                mk[t * m.d + k] = __bfloat162float(kb1);
                mk[t * m.d + k + hd] = __bfloat162float(kb2);
                mk[1024 + t * m.d + k] = __bfloat162float(vb1);
                mk[1024 + t * m.d + k + hd] = __bfloat162float(vb2);
            }
        } else {
            float *kp = reinterpret_cast<float *>(c.p->kpool[l]) + off;
            float *vp = reinterpret_cast<float *>(c.p->vpool[l]) + off;
            kp[k] = k1;
            kp[k + hd] = k2;
            vp[k] = v1;
            vp[k + hd] = v2;
            float *mk = reinterpret_cast<float *>(mini);
            mk[t * m.d + k] = k1;
            mk[t * m.d + k + hd] = k2;
            mk[1024 + t * m.d + k] = v1;
            mk[1024 + t * m.d + k + hd] = v2;
        }
    }
}

// tensor-core attention state of one warp (16 query rows, d = 128)
struct AttMma {
    uint32_t qf[8][4];
    float o[16][4];
    float mrow[2], lrow[2];
};

// one key page: kbase/vbase hold [2 boxes][nkeys][128 B] swizzled, box stride bs
__device__ void att_page_mma(const Ctx &c, AttMma &A, uint32_t kbase, uint32_t vbase, int bs,
                             int nnt, int key_base, int valid, bool causal, int mt, int G) {
    const int r = c.lane >> 2, q = c.lane & 3;
    const float sl2 = rsqrtf((float)c.m->d) * 1.4426950408889634f;
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        if (nt < nnt) {
#pragma unroll
            for (int kk2 = 0; kk2 < 4; ++kk2) {
                int key = 8 * nt + (c.lane & 7);
                int dch = 4 * kk2 + (c.lane >> 3);
                uint32_t ad = kbase + (dch >> 3) * bs + key * 128 + (((dch & 7) ^ (key & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldsm4(ad, b0, b1, b2, b3);
                mma_bf16(sc[nt], A.qf[2 * kk2][0], A.qf[2 * kk2][1], A.qf[2 * kk2][2], A.qf[2 * kk2][3], b0, b1);
                mma_bf16(sc[nt], A.qf[2 * kk2 + 1][0], A.qf[2 * kk2 + 1][1], A.qf[2 * kk2 + 1][2],
                         A.qf[2 * kk2 + 1][3], b2, b3);
            }
        }
    }
    // mask, scale, online softmax (log2 domain)
    float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int key = 8 * nt + 2 * q + (i & 1);
            int row = mt * 16 + r + (i >> 1) * 8;
            bool ok = nt < nnt && key < valid;
            if (causal) ok = ok && key <= row / G;
            float v = ok ? sc[nt][i] * sl2 : -CUDART_INF_F;
            sc[nt][i] = v;
            mx[i >> 1] = fmaxf(mx[i >> 1], v);
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    }
    float corr[2], mn[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        mn[h] = fmaxf(A.mrow[h], mx[h]);
        corr[h] = exp2f(A.mrow[h] - mn[h]);
        A.mrow[h] = mn[h];
        A.lrow[h] *= corr[h];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float p = exp2f(sc[nt][i] - mn[i >> 1]);
            sc[nt][i] = p;
            A.lrow[i >> 1] += p;
        }
    }
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        A.o[nd][0] *= corr[0];
        A.o[nd][1] *= corr[0];
        A.o[nd][2] *= corr[1];
        A.o[nd][3] *= corr[1];
    }
    // P V
    const bool partial = valid < 8 * nnt;
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
        if (2 * kk2 < nnt) {
            uint32_t a0 = pack_bf16(sc[2 * kk2][0], sc[2 * kk2][1]);
            uint32_t a1 = pack_bf16(sc[2 * kk2][2], sc[2 * kk2][3]);
            uint32_t a2 = pack_bf16(sc[2 * kk2 + 1][0], sc[2 * kk2 + 1][1]);
            uint32_t a3 = pack_bf16(sc[2 * kk2 + 1][2], sc[2 * kk2 + 1][3]);
            const int klo = 16 * kk2 + 2 * q;  // keys of b0/b2 halves: klo, klo+1; b1/b3: klo+8, +9
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                int key = 16 * kk2 + (c.lane & 7) + ((c.lane >> 3) & 1) * 8;
                int dch = 2 * np + (c.lane >> 4);
                uint32_t ad = vbase + (dch >> 3) * bs + key * 128 + (((dch & 7) ^ (key & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldsm4t(ad, b0, b1, b2, b3);
                if (partial) {
                    uint32_t m0 = (klo < valid ? 0xffffu : 0u) | (klo + 1 < valid ? 0xffff0000u : 0u);
                    uint32_t m1 = (klo + 8 < valid ? 0xffffu : 0u) | (klo + 9 < valid ? 0xffff0000u : 0u);
                    b0 &= m0;
                    b2 &= m0;
                    b1 &= m1;
                    b3 &= m1;
                }
                mma_bf16(A.o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_bf16(A.o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
}

// FFMA attention of one page for <= 16 rows (fp32 caches, head_dim 64)
struct AttF {
    float o[16][4];
    float mrow[16], lrow[16];
};
__device__ void att_page_f32(const Ctx &c, AttF &A, const float *qs, int R, int G,
                             const unsigned char *kb, const unsigned char *vb, int bs, int es,
                             bool plain, int key0, int nkeys, int valid, bool causal) {
    const DModel &m = *c.m;
    const int nd = m.d / 32;
    const float sl2 = rsqrtf((float)m.d) * 1.4426950408889634f;
    for (int key = key0; key < key0 + nkeys; ++key) {
        if (key >= valid) break;
        float kv[4], vv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            kv[i] = vv[i] = 0.f;
            if (i < nd) {
                int dd = c.lane + 32 * i;
                if (plain) {
                    kv[i] = reinterpret_cast<const float *>(kb)[key * m.d + dd];
                    vv[i] = reinterpret_cast<const float *>(vb)[key * m.d + dd];
                } else {
                    int byte = dd * es;
                    uint32_t off = (byte >> 7) * bs + (swz(0, key, byte & 127));
                    if (es == 4) {
                        kv[i] = *reinterpret_cast<const float *>(kb + off);
                        vv[i] = *reinterpret_cast<const float *>(vb + off);
                    } else {
                        kv[i] = bf16_to_f(*reinterpret_cast<const uint16_t *>(kb + off));
                        vv[i] = bf16_to_f(*reinterpret_cast<const uint16_t *>(vb + off));
                    }
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            if (rr < R) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (i < nd) s += qs[rr * m.d + c.lane + 32 * i] * kv[i];
#pragma unroll
                for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (causal && key > rr / G) continue;
                s *= sl2;
                float mn = fmaxf(A.mrow[rr], s);
                float corr = exp2f(A.mrow[rr] - mn), p = exp2f(s - mn);
                A.mrow[rr] = mn;
                A.lrow[rr] = A.lrow[rr] * corr + p;
#pragma unroll
                for (int i = 0; i < 4; ++i) A.o[rr][i] = A.o[rr][i] * corr + p * vv[i];
            }
        }
    }
}

__device__ bool cons_att(Ctx &c, int l, uint32_t &ci) {
    const DModel &m = *c.m;
    const AttUnit u = att_unit(c);
    const int G = m.Hq / m.Hkv, R = G * c.T;
    const bool mma_path = (m.kv_es == 2 && m.d == 128);
    const int nbox = (m.d * m.kv_es) / 128, bs = m.P * 128;
    const int D2 = m.d + 2;
    compute_inv_rms(c, 0);
    bar_consumers();
    if (u.active) att_prepare(c, l, u, mma_path);
    bar_consumers();
    unsigned char *scr = c.sm + SM_SCRATCH;
    float *part = m.att_part + (long long)(u.g * MK_MAXSPLIT + u.s) * MK_MAXROWS * D2;
    if (u.active && mma_path) {
        const int nmt = (R + 15) / 16, nws = MK_NCWARPS / nmt;
        const int mt = c.warp % nmt, ws = c.warp / nmt;
        const bool wact = c.warp < nmt * nws;
        AttMma A;
        A.mrow[0] = A.mrow[1] = -1e30f;
        A.lrow[0] = A.lrow[1] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) A.o[i][0] = A.o[i][1] = A.o[i][2] = A.o[i][3] = 0.f;
        if (wact) {
            const uint32_t qs = sa(scr);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                int row = mt * 16 + (c.lane & 7) + ((c.lane >> 3) & 1) * 8;
                int col = 16 * kk + (c.lane >> 4) * 8;
                ldsm4(qs + row * 272 + col * 2, A.qf[kk][0], A.qf[kk][1], A.qf[kk][2], A.qf[kk][3]);
            }
        }
        for (int j = u.p0; j < u.pc1; ++j) {
            const int ks = ci % MK_RING, vs = (ci + 1) % MK_RING;
            bool ok = mbar_wait(&c.full[ks], (ci / MK_RING) & 1, c, 210);
            ok = mbar_wait(&c.full[vs], ((ci + 1) / MK_RING) & 1, c, 211) && ok;
            if (ok && wact && ((j - u.p0) % nws) == ws) {
                int valid = min(m.P, c.ctx - j * m.P);
                att_page_mma(c, A, sa(c.sm + SM_RING + ks * MK_SLOT), sa(c.sm + SM_RING + vs * MK_SLOT),
                             bs, 8, j * m.P, valid, false, mt, G);
            }
            __syncwarp();
            if (c.lane == 0) {
                mbar_arrive(&c.empty[ks]);
                mbar_arrive(&c.empty[vs]);
            }
            ci += 2;
        }
        if (u.has_new && wact && ((u.pc1 - u.p0) % nws) == ws) {
            uint32_t mini = sa(scr + 17408);
            att_page_mma(c, A, mini, mini + 4096, 2048, 2, 0, c.T, true, mt, G);
        }
        // finish row sums
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            A.lrow[h] += __shfl_xor_sync(0xffffffffu, A.lrow[h], 1);
            A.lrow[h] += __shfl_xor_sync(0xffffffffu, A.lrow[h], 2);
        }
        bar_consumers();
        // merge the warp streams of each m-tile through scratch
        const int r = c.lane >> 2, q = c.lane & 3;
        float *mrg = reinterpret_cast<float *>(scr);
        const int WS = 16 * 128 + 32;
        if (wact && ws > 0) {
            float *w = mrg + ((ws - 1) * nmt + mt) * WS;
#pragma unroll
            for (int nd = 0; nd < 16; ++nd) {
                w[r * 128 + nd * 8 + 2 * q] = A.o[nd][0];
                w[r * 128 + nd * 8 + 2 * q + 1] = A.o[nd][1];
                w[(r + 8) * 128 + nd * 8 + 2 * q] = A.o[nd][2];
                w[(r + 8) * 128 + nd * 8 + 2 * q + 1] = A.o[nd][3];
            }
            if (q == 0) {
                w[2048 + r] = A.mrow[0];
                w[2048 + r + 8] = A.mrow[1];
                w[2064 + r] = A.lrow[0];
                w[2064 + r + 8] = A.lrow[1];
            }
        }
        bar_consumers();
        if (wact && ws == 0) {
            for (int o2 = 1; o2 < nws; ++o2) {
                const float *w = mrg + ((o2 - 1) * nmt + mt) * WS;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    int rr = r + 8 * h;
                    float m2 = w[2048 + rr], l2 = w[2064 + rr];
                    float mn = fmaxf(A.mrow[h], m2);
                    float a = exp2f(A.mrow[h] - mn), b = exp2f(m2 - mn);
                    A.mrow[h] = mn;
                    A.lrow[h] = A.lrow[h] * a + l2 * b;
#pragma unroll
                    for (int nd = 0; nd < 16; ++nd) {
                        A.o[nd][2 * h] = A.o[nd][2 * h] * a + w[rr * 128 + nd * 8 + 2 * q] * b;
                        A.o[nd][2 * h + 1] = A.o[nd][2 * h + 1] * a + w[rr * 128 + nd * 8 + 2 * q + 1] * b;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int row = mt * 16 + r + 8 * h;
                if (row < R) {
                    float *dst = part + row * D2;
#pragma unroll
                    for (int nd = 0; nd < 16; ++nd)
                        __stcg(reinterpret_cast<float2 *>(dst + nd * 8 + 2 * q),
                               make_float2(A.o[nd][2 * h], A.o[nd][2 * h + 1]));
                    if (q == 0) {
                        __stcg(dst + m.d, A.mrow[h]);
                        __stcg(dst + m.d + 1, A.lrow[h]);
                    }
                }
            }
        }
    } else if (u.active) {
        // FFMA path: all warps share every page, each warp takes 8 keys
        AttF A;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            A.mrow[rr] = -1e30f;
            A.lrow[rr] = 0.f;
            A.o[rr][0] = A.o[rr][1] = A.o[rr][2] = A.o[rr][3] = 0.f;
        }
        const float *qs = reinterpret_cast<const float *>(scr);
        const int kpw = m.P / MK_NCWARPS;
        for (int j = u.p0; j < u.pc1; ++j) {
            const int ks = ci % MK_RING, vs = (ci + 1) % MK_RING;
            bool ok = mbar_wait(&c.full[ks], (ci / MK_RING) & 1, c, 212);
            ok = mbar_wait(&c.full[vs], ((ci + 1) / MK_RING) & 1, c, 213) && ok;
            if (ok) {
                int valid = min(m.P, c.ctx - j * m.P);
                att_page_f32(c, A, qs, R, G, c.sm + SM_RING + ks * MK_SLOT, c.sm + SM_RING + vs * MK_SLOT,
                             bs, m.kv_es, false, c.warp * kpw, kpw, valid, false);
            }
            __syncwarp();
            if (c.lane == 0) {
                mbar_arrive(&c.empty[ks]);
                mbar_arrive(&c.empty[vs]);
            }
            ci += 2;
        }
        if (u.has_new && c.warp == 0) {
            const unsigned char *mini = scr + 17408;
            att_page_f32(c, A, qs, R, G, mini, mini + 4096, 0, 4, true, 0, c.T, c.T, true);
        }
        bar_consumers();
        float *mrg = reinterpret_cast<float *>(scr);
        const int WS = 16 * m.d + 32, MO = 16 * m.d;
        float *w = mrg + c.warp * WS;
        const int nd = m.d / 32;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            if (rr < R) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (i < nd) w[rr * m.d + c.lane + 32 * i] = A.o[rr][i];
                if (c.lane == 0) {
                    w[MO + rr] = A.mrow[rr];
                    w[MO + 16 + rr] = A.lrow[rr];
                }
            }
        }
        bar_consumers();
        for (int i = c.tid; i < R * m.d; i += MK_NCWARPS * 32) {
            int rr = i / m.d, dd = i - rr * m.d;
            float mn = -1e30f;
            for (int o2 = 0; o2 < MK_NCWARPS; ++o2) mn = fmaxf(mn, mrg[o2 * WS + MO + rr]);
            float acc = 0.f, lsum = 0.f;
            for (int o2 = 0; o2 < MK_NCWARPS; ++o2) {
                float a = exp2f(mrg[o2 * WS + MO + rr] - mn);
                acc += a * mrg[o2 * WS + rr * m.d + dd];
                lsum += a * mrg[o2 * WS + MO + 16 + rr];
            }
            float *dst = part + rr * D2;
            __stcg(dst + dd, acc);
            if (dd == 0) {
                __stcg(dst + m.d, mn);
                __stcg(dst + m.d + 1, lsum);
            }
        }
    }
    // group barrier among the splits of this kv head, then merge assigned rows
    bar_consumers();
    if (!u.active) return true;
    if (c.tid == 0) {
        bool ok = !aborted(c);
        __threadfence();
        atomicAdd(m.att_cnt + l * m.Hkv + u.g, 1);
        if (ok) ok = spin_ge_s32(m.att_cnt + l * m.Hkv + u.g, c.nsplit, c, 220);
        __threadfence();
        c.misc->gs_ok = ok;
    }
    bar_consumers();
    if (!c.misc->gs_ok) return false;
    int r0, r1;
    split_range(R, c.nsplit, u.s, r0, r1);
    const float *pbase = m.att_part + (long long)(u.g * MK_MAXSPLIT) * MK_MAXROWS * D2;
    for (int i = c.tid; i < (r1 - r0) * m.d; i += MK_NCWARPS * 32) {
        int row = r0 + i / m.d, dd = i % m.d;
        float mn = -1e30f;
        for (int s = 0; s < c.nsplit; ++s) mn = fmaxf(mn, __ldcg(pbase + ((long long)s * MK_MAXROWS + row) * D2 + m.d));
        float acc = 0.f, lsum = 0.f;
        for (int s = 0; s < c.nsplit; ++s) {
            const float *pp = pbase + ((long long)s * MK_MAXROWS + row) * D2;
            float a = exp2f(__ldcg(pp + m.d) - mn);
            acc += a * __ldcg(pp + dd);
            lsum += a * __ldcg(pp + m.d + 1);
        }
        int t = row / G, h = u.g * G + (row - t * G);
        __stcg(m.o_buf + (long long)t * m.Hq * m.d + h * m.d + dd, acc / lsum);
    }
    return true;
}

// ------------------------------------------------------------------ consumer
__device__ void consumer(Ctx &c) {
    const DModel &m = *c.m;
    const Params &p = *c.p;
    uint32_t ci = 0;
    const bool f32path = m.wdt == MK_DT_F32;
    const uint32_t allH = 0xffffffffu >> (32 - m.H / 128);
    int nl = p.mode ? 1 : m.L;
    // zero the accumulators, load the residual stream
    zero_slice(c, m.qkv_acc, (long long)MK_MAXT * m.nqkv);
    zero_slice(c, m.sh_acc, (long long)MK_MAXT * 2 * m.I);
    zero_slice(c, m.ea_acc, (long long)MK_MAXT * m.K * 2 * m.I);
    zero_slice(c, m.rlog, (long long)MK_MAXT * m.E);
    if (p.mode == 0) zero_slice(c, m.logit_acc, (long long)c.T * m.V);
    if (c.cta == 0)
        for (int i = c.tid; i < m.L * m.Hkv; i += MK_NCWARPS * 32) __stcg(m.att_cnt + i, 0);
    {
        long long n = (long long)c.T * m.H;
        long long b = n * c.cta / c.G, e = n * (c.cta + 1) / c.G;
        for (long long i = b + c.tid; i < e; i += MK_NCWARPS * 32) {
            int t = (int)(i / m.H), col = (int)(i - (long long)t * m.H);
            float v = p.mode ? __ldg(p.hidden_in + i)
                             : bf16_to_f(__ldg(m.embed + (long long)__ldg(p.tokens + t) * m.H + col));
            __stcg(m.res + (long long)t * m.H + col, to_fx(v));
        }
    }
    if (!grid_sync(c, 1)) return;
    for (int li = 0; li < nl; ++li) {
        const int l = p.mode ? p.layer : li;
        const DLayer &L = m.layers[l];
        RouteSm *rt = &c.rt[li & 1];
        // ---- QKV
        {
            ActSrc a{m.res, nullptr, m.H, L.attn_norm};
            int b, e;
            split_range(stage_total(m, ST_QKV, L, rt), c.G, c.cta, b, e);
            if (f32path) build_act32(c, a, m.H);
            else build_frags(c, a, needed_kb(b, e, L.qkv));
            ssq_block(c, 0);
            zero_slice(c, m.sh_acc, (long long)MK_MAXT * 2 * m.I);
            zero_slice(c, m.ea_acc, (long long)MK_MAXT * m.K * 2 * m.I);
            bar_consumers();
            cons_gemv(c, ST_QKV, L, rt, ci);
            if (!grid_sync(c, 2)) return;
        }
        // ---- attention
        if (!cons_att(c, l, ci)) return;
        if (!grid_sync(c, 3)) return;
        // ---- O projection (+ residual)
        {
            ActSrc a{nullptr, m.o_buf, m.Hq * m.d, nullptr};
            int b, e;
            split_range(stage_total(m, ST_O, L, rt), c.G, c.cta, b, e);
            if (f32path) build_act32(c, a, m.Hq * m.d);
            else build_frags(c, a, needed_kb(b, e, L.o));
            zero_slice(c, m.qkv_acc, (long long)MK_MAXT * m.nqkv);
            bar_consumers();
            cons_gemv(c, ST_O, L, rt, ci);
            if (!grid_sync(c, 4)) return;
        }
        // ---- router + shared expert gate/up, then routed gate/up
        {
            ActSrc a{m.res, nullptr, m.H, L.moe_norm};
            if (f32path) build_act32(c, a, m.H);
            else build_frags(c, a, allH);
            ssq_block(c, 1);
            bar_consumers();
            cons_gemv(c, ST_ROUTER, L, rt, ci);
            grid_arrive(c);
            cons_gemv(c, ST_SHA, L, rt, ci);
            if (!grid_wait(c, 5)) return;
            compute_inv_rms(c, 1);
            bar_consumers();
            route_layer(c, L, rt);
            if (c.tid == 0) mbar_arrive(c.route);
            if (c.cta == 0) {
                if (c.tid == 0) c.misc->distinct_total += rt->nd;
                if (p.mode == 1) {
                    for (int i = c.tid; i < c.T * m.K; i += MK_NCWARPS * 32) {
                        if (p.out_idx) p.out_idx[i] = rt->idx[i / m.K][i % m.K];
                        if (p.out_w) p.out_w[i] = rt->w[i / m.K][i % m.K];
                    }
                } else if (p.trace) {
                    for (int i = c.tid; i < c.T * m.K; i += MK_NCWARPS * 32)
                        p.trace[(long long)l * c.T * m.K + i] = rt->idx[i / m.K][i % m.K];
                }
            }
            cons_gemv(c, ST_EXPA, L, rt, ci);
            if (!grid_sync(c, 6)) return;
        }
        // ---- routed + shared down projections (+ residual)
        zero_slice(c, m.rlog, (long long)MK_MAXT * m.E);
        cons_gemv(c, ST_EXPB, L, rt, ci);
        if (!grid_sync(c, 7)) return;
    }
    if (p.mode == 1) {
        long long n = (long long)c.T * m.H;
        long long b = n * c.cta / c.G, e = n * (c.cta + 1) / c.G;
        for (long long i = b + c.tid; i < e; i += MK_NCWARPS * 32) p.hidden_out[i] = from_fx(__ldcg(m.res + i));
        if (c.cta == 0 && c.tid == 0) c.ctrl->epoch = c.bar_base + (unsigned long long)c.nbar * c.G;
        return;
    }
    // ---- final norm + LM head
    {
        ActSrc a{m.res, nullptr, m.H, m.final_norm};
        build_frags(c, a, allH);
        ssq_block(c, 2);
        bar_consumers();
        cons_gemv(c, ST_LM, m.layers[0], &c.rt[0], ci);
        if (!grid_sync(c, 8)) return;
    }
    // ---- logits, per-CTA argmax candidates
    compute_inv_rms(c, 2);
    bar_consumers();
    {
        float *bv = reinterpret_cast<float *>(c.sm + SM_SCRATCH);
        int *bi = reinterpret_cast<int *>(c.sm + SM_SCRATCH + 4096);
        int b, e;
        split_range(m.V, c.G, c.cta, b, e);
        for (int t = 0; t < c.T; ++t) {
            float inv = c.misc->inv_rms[2][t];
            float best = -CUDART_INF_F;
            int besti = 0x7fffffff;
            for (int v = b + c.tid; v < e; v += MK_NCWARPS * 32) {
                float lg = from_fx(__ldcg(m.logit_acc + (long long)t * m.V + v)) * inv;
                p.out_logits[(long long)t * m.V + v] = lg;
                if (lg > best || (lg == best && v < besti)) {
                    best = lg;
                    besti = v;
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                float ob = __shfl_xor_sync(0xffffffffu, best, o);
                int oi = __shfl_xor_sync(0xffffffffu, besti, o);
                if (ob > best || (ob == best && oi < besti)) {
                    best = ob;
                    besti = oi;
                }
            }
            if (c.lane == 0) {
                bv[t * 8 + c.warp] = best;
                bi[t * 8 + c.warp] = besti;
            }
        }
        bar_consumers();
        if (c.tid < c.T) {
            int t = c.tid;
            float best = -CUDART_INF_F;
            int besti = 0x7fffffff;
            for (int w = 0; w < MK_NCWARPS; ++w) {
                float ob = bv[t * 8 + w];
                int oi = bi[t * 8 + w];
                if (ob > best || (ob == best && oi < besti)) {
                    best = ob;
                    besti = oi;
                }
            }
            __stcg(m.cand_v + c.cta * MK_MAXT + t, best);
            __stcg(m.cand_i + c.cta * MK_MAXT + t, besti);
        }
    }
    if (!grid_sync(c, 9)) return;
    if (c.cta == 0) {
        int *am = reinterpret_cast<int *>(c.sm + SM_SCRATCH + 8192);
        if (c.tid < c.T) {
            int t = c.tid;
            float best = -CUDART_INF_F;
            int besti = 0x7fffffff;
            for (int k = 0; k < c.G; ++k) {
                float ob = __ldcg(m.cand_v + k * MK_MAXT + t);
                int oi = __ldcg(m.cand_i + k * MK_MAXT + t);
                if (ob > best || (ob == best && oi < besti)) {
                    best = ob;
                    besti = oi;
                }
            }
            am[t] = besti;
            if (p.out_argmax) p.out_argmax[t] = besti;
        }
        bar_consumers();
        if (c.tid == 0) {
            int n = 0;
            for (int i = 1; i < c.T; ++i) {
                if (__ldg(p.tokens + i) == am[i - 1]) n = i;
                else break;
            }
            *p.out_accepted = n;
            Ctrl *k = c.ctrl;
            k->steps += 1;
            k->accepted_sum += n;
            k->distinct_sum += c.misc->distinct_total;
            k->last_accepted = n;
            k->last_distinct = c.misc->distinct_total;
            k->epoch = c.bar_base + (unsigned long long)c.nbar * c.G;
        }
    }
}

__global__ void __launch_bounds__(MK_THREADS, 1) mk_step_kernel(const __grid_constant__ Params p) {
    extern __shared__ unsigned char smem_raw[];
    // the 128-byte TMA swizzle pattern repeats every 1024 bytes: align the map to it
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Ctx c;
    c.p = &p;
    c.m = p.m;
    c.ctrl = p.m->ctrl;
    c.sm = smem;
    c.full = reinterpret_cast<uint64_t *>(smem + SM_BAR);
    c.empty = c.full + MK_RING;
    c.route = c.empty + MK_RING;
    c.rt = reinterpret_cast<RouteSm *>(smem + SM_ROUTE);
    c.misc = reinterpret_cast<MiscSm *>(smem + SM_MISC);
    c.cta = blockIdx.x;
    c.G = gridDim.x;
    c.T = p.T;
    c.tid = threadIdx.x;
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    c.nbar = 0;
    c.timeout = p.m->timeout_ns;
    const DModel &m = *p.m;
    if (threadIdx.x == 0) {
        for (int i = 0; i < MK_RING; ++i) {
            mbar_init(&c.full[i], 1);
            mbar_init(&c.empty[i], MK_NCWARPS);
        }
        mbar_init(c.route, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        c.misc->abort = 0;
        c.misc->distinct_total = 0;
        // validate the step's inputs (every CTA reaches the same verdict)
        int ctx = __ldg(p.positions);
        int ok = (*(volatile int *)&c.ctrl->abort == 0) ? 1 : 0;
        for (int t = 0; t < p.T; ++t)
            if (__ldg(p.positions + t) != ctx + t) ok = 0;
        if (ctx < 0 || (long long)ctx + p.T > (long long)m.max_pages * m.P) ok = 0;
        if (ok) {
            int np = (ctx + p.T + m.P - 1) / m.P;
            for (int j = 0; j < np; ++j) {
                int ph = __ldg(p.page_table + j);
                if (ph < 0 || ph >= p.n_pages) ok = 0;
            }
        }
        if (ok && p.mode == 0) {
            for (int t = 0; t < p.T; ++t) {
                int tk = __ldg(p.tokens + t);
                if (tk < 0 || tk >= m.V) ok = 0;
            }
        }
        c.misc->valid = ok;
        c.misc->ctx = ctx;
        c.misc->base = *(volatile unsigned long long *)&c.ctrl->epoch;
    }
    __syncthreads();
    if (!c.misc->valid) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && *(volatile int *)&c.ctrl->abort == 0) {
            atomicCAS(&c.ctrl->status, 0, (int)MK_ERR_BAD_INPUT);
            atomicExch(&c.ctrl->abort, 1);
        }
        return;
    }
    c.ctx = c.misc->ctx;
    c.bar_base = c.misc->base;
    {
        int ncp = (c.ctx + m.P - 1) / m.P;
        c.nsplit = min(min(c.G / m.Hkv, ncp + 1), MK_MAXSPLIT);
    }
    if (c.warp == MK_NCWARPS) {
        if (c.lane == 0) producer(c);
        __syncwarp();
    } else {
        consumer(c);
    }
}

}  // namespace

cudaError_t mk_kernel_setup(size_t smem) {
    return cudaFuncSetAttribute(mk_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t mk_launch(const Params &p, int grid, size_t smem, cudaStream_t s) {
    void *args[] = {(void *)&p};
    return cudaLaunchCooperativeKernel((const void *)mk_step_kernel, dim3(grid), dim3(MK_THREADS), args, smem, s);
}

int mk_kernel_max_blocks(size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mk_step_kernel, MK_THREADS, smem) != cudaSuccess) return -1;
    return n;
}
