// Gated DeltaNet decode, the state kernels (gdn_decode_step and the fused
// conv + GDN layer) as one persistent, warp-specialised TMA pipeline for
// sm_103a.
//
// The step is state traffic: every real (row, value head) reads a dv x dk
// fp32 state and writes the next one, with a few multiply-adds per element
// ("mstar PR #1139", section "Why": a kernel with the same reads and writes
// and no math takes 45.2 of the rule's 46.1 us).  The kernel therefore keeps
// as many bytes in flight as shared memory allows and spends as few
// instructions as possible per byte:
//
//  * Work item = RB consecutive value rows of one (row, value head): 16 KiB of
//    fp32 state (RB = 4096 / dk), contiguous in the pool.  Items are dealt
//    round-robin to two CTAs per SM (persistent grid), so every CTA gets the
//    same number of items to within one.
//  * Producer warp: prepares items 32 at a time (each lane loads one item's
//    slots and gate inputs and computes its gates), then one lane copies each
//    item's metadata into a free stage and issues cp.async.bulk copies of the
//    state chunk and
//    of the item's small inputs (q, k, v -- or, in the fused layer, the conv
//    windows, tokens, taps and bias of the item's channels) into a ring of
//    shared-memory stages, completing on the stage's "full" mbarrier.
//  * Consumer warps (8): per item, the prologue computes the q/k/v values
//    (the conv in the fused layer) and the L2 norms by a block reduction among
//    consumers; then each lane owns 16 floats of one state row
//    (dk/16 lanes a row, 16-byte vectors interleaved so a warp store covers
//    whole 128-byte lines), forms u = S k^ and w = S q^ in one butterfly, and
//    stores S' = alpha S + c k^ (c = beta (v - alpha u)) straight to HBM with
//    o = alpha w + c (k^ . q^).  Then the warps release the stage ("empty").
//  * Every wait is bounded: a wait that runs out reports GDN_DEVERR_TIMEOUT,
//    the consumers agree on it through a barrier reduction, and the CTA stops
//    after the producer has waited (bounded) for its copies still in flight.
//
// Fused layer, in place: the q/k conv window of a qk group is read by every
// item of the group and must be written once, after all of them read it.
// In-place launches deal whole groups (all value heads and row chunks sharing
// the qk head) to one CTA, in order, and the group's last item writes the
// window.  Twin launches write another slot, so the chunk-0 item of the
// group's first value head writes it at once.  The arithmetic per row is the
// same in every schedule, so twin and in place give bit-identical values.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32; // + one producer warp
constexpr float kL2Eps = 1e-6f;
constexpr int kBarId = 1;                 // named barrier among the consumers
constexpr long long kWaitLimit = 1ll << 20;
constexpr int kCtasPerSm = 2;

template <int DK> struct Geo {
    static_assert(DK >= 16 && DK <= 256 && DK % 16 == 0, "dk");
    static constexpr int LPR = DK / 16;              // lanes per state row
    static constexpr int RPW = 32 / LPR;             // state rows per warp
    static constexpr int RB = RPW * kConsumerWarps;  // state rows per item (4096 / DK)
};

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, bulk copy, named barrier with an OR reduction
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sm_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Bounded wait for the phase of `parity` to complete; false when it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    for (long long i = 0; i < kWaitLimit; ++i)
        if (mbar_try(bar, parity))
            return true;
    return false;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// Named barrier over the consumer warps that also ORs a predicate across them.
__device__ __forceinline__ bool consumers_sync_or(bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "n"(kBarId), "n"(kConsumers)
                 : "memory");
    return r != 0;
}

template <typename T>
__device__ __forceinline__ float ld_act(const void *base, size_t idx)
{
    return to_f(reinterpret_cast<const T *>(base)[idx]);
}
template <typename T>
__device__ __forceinline__ float sh_act(const unsigned char *base, int idx)
{
    return to_f(reinterpret_cast<const T *>(base)[idx]);
}

// ---------------------------------------------------------------------------
// Shared-memory stage layout (byte offsets, all 16-byte aligned)
// ---------------------------------------------------------------------------
template <typename T, int DK, bool LAYER, int W> struct Stage {
    static constexpr int RB = Geo<DK>::RB;
    static constexpr int E = sizeof(T);
    static constexpr int NCH = 2 * DK + RB;            // channels an item needs (q | k | v)
    static constexpr int align16(int x) { return (x + 15) & ~15; }
    static constexpr int STATE = 0;
    static constexpr int STATE_BYTES = RB * DK * 4;
    // raw inputs (TMA destinations)
    static constexpr int RAW = STATE + STATE_BYTES;
    // step:  q[DK] | k[DK] | v[RB]
    // layer: win[W-1][NCH] | x[NCH] | w[NCH][W] | bias[NCH], each [q | k | v]
    static constexpr int WIN = RAW;
    static constexpr int XS = LAYER ? WIN + (W - 1) * NCH * E : RAW;
    static constexpr int WS = XS + NCH * E;
    static constexpr int BS = WS + NCH * W * E;
    static constexpr int RAW_END = LAYER ? BS + NCH * E : RAW + NCH * E;
    // computed by the consumers
    static constexpr int QN = align16(RAW_END);        // q values (fp32) [DK]
    static constexpr int KN = QN + DK * 4;             // k values (fp32) [DK]
    static constexpr int VN = KN + DK * 4;             // v values (fp32) [RB]
    static constexpr int PART = VN + RB * 4;           // block-reduction partials [3][8]
    static constexpr int META = align16(PART + 3 * kConsumerWarps * 4); // Meta, by the producer
    static constexpr int BYTES = (META + 48 + 127) & ~127;
};

struct Meta {
    int r, h, chunk, rs, ws, live, last, rows;
    float alpha, beta;
};

// The item sequence of one CTA.  Fine: items dealt round-robin.  Coarse:
// whole qk groups dealt round-robin, the items of a group in order.
struct Sched {
    int hv, group, chunks;
    int n_units;     // items (fine) or groups (coarse)
    int per_unit;    // 1 (fine) or group * chunks (coarse)
    int coarse;

    // number of items CTA b of a grid of g CTAs processes
    __device__ __forceinline__ int count(int b, int g) const
    {
        if (b >= n_units)
            return 0;
        return ((n_units - 1 - b) / g + 1) * per_unit;
    }

    // k-th item of CTA b in a grid of g CTAs (k < count(b, g))
    __device__ __forceinline__ void item(int b, int g, int k, int &r, int &h, int &chunk, bool &last) const
    {
        const int unit = b + (k / per_unit) * g;
        if (!coarse) {
            chunk = unit % chunks;
            const int rh = unit / chunks;
            h = rh % hv;
            r = rh / hv;
            last = false;
        } else {
            const int j = k % per_unit;
            const int hk = hv / group;
            r = unit / hk;
            h = (unit % hk) * group + j / chunks;
            chunk = j % chunks;
            last = j == per_unit - 1;
        }
    }
};

template <typename T, int DK, bool LAYER, int W>
__global__ void __launch_bounds__(kThreads, 2) gdn_stream_kernel(const StepArgs p, const Sched sc, int nstages)
{
    using G = Geo<DK>;
    using L = Stage<T, DK, LAYER, W>;
    constexpr int RB = G::RB;
    constexpr int E = L::E;

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bars[2 * 8]; // full[s], empty[s]
    __shared__ int abort_flag;
    __shared__ int issued_n, consumed_n;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nst = nstages;
    auto full_bar = [&](int s) { return sm_addr(&bars[s]); };
    auto empty_bar = [&](int s) { return sm_addr(&bars[8 + s]); };
    auto stage = [&](int s) { return smem + (size_t)s * L::BYTES; };

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        abort_flag = 0;
        issued_n = 0;
        consumed_n = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int C = p.channels;
    if (warp == kConsumerWarps) {
        // =========================== producer ===========================
        // The warp prepares items 32 at a time: lane j loads item j's slots
        // and gate inputs (independent loads, all in flight together) and
        // computes its gates into a shared table; lane 0 then streams the
        // batch: wait for a free stage, copy the item's metadata into it, issue
        // the bulk copies.
        __shared__ Meta table[32];
        const int n_items = sc.count(blockIdx.x, gridDim.x);
        bool stop = false;
        for (int base = 0; base < n_items && !stop; base += 32) {
            const int kk = base + lane;
            if (kk < n_items) {
                Meta q;
                bool last;
                sc.item(blockIdx.x, gridDim.x, kk, q.r, q.h, q.chunk, last);
                q.last = last;
                q.rs = p.read_slot[q.r];
                q.ws = p.in_place ? q.rs : p.write_slot[q.r];
                const float av = ld_act<T>(p.a, (size_t)q.r * p.hv + q.h);
                const float bv = ld_act<T>(p.b, (size_t)q.r * p.hv + q.h);
                const float al = p.A_log[q.h], dt = p.dt_bias[q.h];
                const int cls = classify_row(q.rs, q.ws, p.num_slots, p.in_place != 0);
                if (cls < 0)
                    report(p.err, GDN_DEVERR_BAD_SLOT);
                q.live = cls == 1;
                q.rows = min(RB, p.dv - q.chunk * RB);
                q.alpha = q.live ? gate_alpha(al, av, dt) : 0.f;
                q.beta = q.live ? gate_beta(bv) : 0.f;
                table[lane] = q;
            }
            __syncwarp();
            if (lane == 0) {
                const int nb = min(32, n_items - base);
                for (int j = 0; j < nb; ++j) {
                    const int k = base + j;
                    const int s = k % nst;
                    const uint32_t par = (uint32_t)((k / nst) & 1);
                    if (!mbar_wait(empty_bar(s), par ^ 1u)) {
                        report(p.err, GDN_DEVERR_TIMEOUT);
                        atomicExch(&abort_flag, 1);
                        stop = true;
                        break;
                    }
                    if (*(volatile int *)&abort_flag) {
                        stop = true;
                        break;
                    }
                    const Meta q = table[j];
                    unsigned char *st = stage(s);
                    *reinterpret_cast<Meta *>(st + L::META) = q;
                    const uint32_t fb = full_bar(s);
                    if (q.live) {
                        const int r = q.r, h = q.h, chunk = q.chunk, rows = q.rows;
                        const int g = h / (p.hv / p.hk);
                        const int cq = g * DK, ck = p.hk * DK + g * DK;
                        const int cv = 2 * p.hk * DK + h * p.dv + chunk * RB;
                        uint32_t bytes = (uint32_t)(rows * DK * 4);
                        if constexpr (LAYER)
                            bytes += (uint32_t)(((W - 1) + 1 + W + (p.bias ? 1 : 0)) * (2 * DK + rows) * E);
                        else
                            bytes += (uint32_t)((2 * DK + rows) * E);
                        mbar_arrive_tx(fb, bytes);
                        const float *src =
                            p.pool + (((size_t)q.rs * p.hv + h) * p.dv + (size_t)chunk * RB) * DK;
                        bulk_load(sm_addr(st + L::STATE), src, (uint32_t)(rows * DK * 4), fb);
                        if constexpr (LAYER) {
                            const unsigned char *conv = reinterpret_cast<const unsigned char *>(p.conv);
                            const unsigned char *x = reinterpret_cast<const unsigned char *>(p.x);
                            const unsigned char *w = reinterpret_cast<const unsigned char *>(p.w);
                            const unsigned char *bias = reinterpret_cast<const unsigned char *>(p.bias);
                            const int off[3] = {0, DK, 2 * DK};
                            const int ch[3] = {cq, ck, cv};
                            const int n[3] = {DK, DK, rows};
#pragma unroll
                            for (int sgm = 0; sgm < 3; ++sgm) {
#pragma unroll
                                for (int jj = 0; jj < W - 1; ++jj)
                                    bulk_load(sm_addr(st + L::WIN + (jj * L::NCH + off[sgm]) * E),
                                              conv + (((size_t)q.rs * (W - 1) + jj) * C + ch[sgm]) * E,
                                              (uint32_t)(n[sgm] * E), fb);
                                bulk_load(sm_addr(st + L::XS + off[sgm] * E), x + ((size_t)r * C + ch[sgm]) * E,
                                          (uint32_t)(n[sgm] * E), fb);
                                bulk_load(sm_addr(st + L::WS + off[sgm] * W * E), w + (size_t)ch[sgm] * W * E,
                                          (uint32_t)(n[sgm] * W * E), fb);
                                if (bias)
                                    bulk_load(sm_addr(st + L::BS + off[sgm] * E), bias + (size_t)ch[sgm] * E,
                                              (uint32_t)(n[sgm] * E), fb);
                            }
                        } else {
                            const unsigned char *qp = reinterpret_cast<const unsigned char *>(p.q);
                            const unsigned char *kp = reinterpret_cast<const unsigned char *>(p.k);
                            const unsigned char *vp = reinterpret_cast<const unsigned char *>(p.v);
                            bulk_load(sm_addr(st + L::RAW), qp + ((size_t)r * p.hk + g) * DK * E, DK * E, fb);
                            bulk_load(sm_addr(st + L::RAW + DK * E), kp + ((size_t)r * p.hk + g) * DK * E,
                                      DK * E, fb);
                            bulk_load(sm_addr(st + L::RAW + 2 * DK * E),
                                      vp + (((size_t)r * p.hv + h) * p.dv + (size_t)chunk * RB) * E,
                                      (uint32_t)(rows * E), fb);
                        }
                    } else {
                        mbar_arrive(fb);
                    }
                    issued_n = k + 1;
                }
            }
            stop = __shfl_sync(0xffffffffu, stop, 0);
            __syncwarp();
        }
    } else {
        // =========================== consumers ==========================
        const int lrow = lane / G::LPR, lcol = lane % G::LPR;
        const int t = tid; // consumer index 0..255
        const int n_items = sc.count(blockIdx.x, gridDim.x);
        for (int k = 0; k < n_items; ++k) {
            const int s = (int)(k % nst);
            const uint32_t par = (uint32_t)((k / nst) & 1);
            const bool got = mbar_wait(full_bar(s), par);
            unsigned char *st = stage(s);
            const Meta m = *reinterpret_cast<const Meta *>(st + L::META);
            const bool live = got && m.live;
            float *qn = reinterpret_cast<float *>(st + L::QN);
            float *kn = reinterpret_cast<float *>(st + L::KN);
            float *vn = reinterpret_cast<float *>(st + L::VN);
            float *part = reinterpret_cast<float *>(st + L::PART);
            T *out = reinterpret_cast<T *>(p.out) + ((size_t)m.r * p.hv + m.h) * p.dv + (size_t)m.chunk * RB;

            // ---- prologue: q, k, v values, norms' partial sums, gates -------
            float pqq = 0.f, pkk = 0.f, pqk = 0.f;
            if (live) {
                const int group = p.hv / p.hk;
                const int g = m.h / group;
                if (t < DK) {
                    float qv, kv;
                    if constexpr (LAYER) {
                        float wq[W], wk[W], winq[W - 1], wink[W - 1];
#pragma unroll
                        for (int j = 0; j < W; ++j) {
                            wq[j] = sh_act<T>(st + L::WS, t * W + j);
                            wk[j] = sh_act<T>(st + L::WS, (DK + t) * W + j);
                        }
#pragma unroll
                        for (int j = 0; j < W - 1; ++j) {
                            winq[j] = sh_act<T>(st + L::WIN, j * L::NCH + t);
                            wink[j] = sh_act<T>(st + L::WIN, j * L::NCH + DK + t);
                        }
                        const float xq = sh_act<T>(st + L::XS, t);
                        const float xk = sh_act<T>(st + L::XS, DK + t);
                        const float bq = p.bias ? sh_act<T>(st + L::BS, t) : 0.f;
                        const float bk = p.bias ? sh_act<T>(st + L::BS, DK + t) : 0.f;
                        qv = round_act<T>(conv_channel<W>(winq, xq, wq, bq, p.silu != 0));
                        kv = round_act<T>(conv_channel<W>(wink, xk, wk, bk, p.silu != 0));
                        // the q/k window is written once per group: by the chunk-0 item
                        // of its first value head (twin), or by its last item (in place)
                        const bool writer = p.in_place ? m.last : (m.h % group == 0 && m.chunk == 0);
                        if (writer) {
                            T *wout = reinterpret_cast<T *>(p.conv) + (size_t)m.ws * (W - 1) * C;
                            const int cq = g * DK + t, ck = p.hk * DK + g * DK + t;
#pragma unroll
                            for (int j = 0; j + 1 < W - 1; ++j) {
                                wout[(size_t)j * C + cq] = from_f<T>(winq[j + 1]);
                                wout[(size_t)j * C + ck] = from_f<T>(wink[j + 1]);
                            }
                            wout[(size_t)(W - 2) * C + cq] = from_f<T>(xq);
                            wout[(size_t)(W - 2) * C + ck] = from_f<T>(xk);
                        }
                    } else {
                        qv = sh_act<T>(st + L::RAW, t);
                        kv = sh_act<T>(st + L::RAW, DK + t);
                    }
                    qn[t] = qv;
                    kn[t] = kv;
                    pqq = qv * qv;
                    pkk = kv * kv;
                    pqk = qv * kv;
                }
                if (t < m.rows) {
                    float vv;
                    if constexpr (LAYER) {
                        float wv[W], winv[W - 1];
#pragma unroll
                        for (int j = 0; j < W; ++j)
                            wv[j] = sh_act<T>(st + L::WS, (2 * DK + t) * W + j);
#pragma unroll
                        for (int j = 0; j < W - 1; ++j)
                            winv[j] = sh_act<T>(st + L::WIN, j * L::NCH + 2 * DK + t);
                        const float xv = sh_act<T>(st + L::XS, 2 * DK + t);
                        const float bv = p.bias ? sh_act<T>(st + L::BS, 2 * DK + t) : 0.f;
                        vv = round_act<T>(conv_channel<W>(winv, xv, wv, bv, p.silu != 0));
                        // this item is the only reader and writer of its v channels
                        T *wout = reinterpret_cast<T *>(p.conv) + (size_t)m.ws * (W - 1) * C;
                        const int cv = 2 * p.hk * DK + m.h * p.dv + m.chunk * RB + t;
#pragma unroll
                        for (int j = 0; j + 1 < W - 1; ++j)
                            wout[(size_t)j * C + cv] = from_f<T>(winv[j + 1]);
                        wout[(size_t)(W - 2) * C + cv] = from_f<T>(xv);
                    } else {
                        vv = sh_act<T>(st + L::RAW, 2 * DK + t);
                    }
                    vn[t] = vv;
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    pqq += __shfl_xor_sync(0xffffffffu, pqq, off);
                    pkk += __shfl_xor_sync(0xffffffffu, pkk, off);
                    pqk += __shfl_xor_sync(0xffffffffu, pqk, off);
                }
                if (lane == 0) {
                    part[0 * kConsumerWarps + warp] = pqq;
                    part[1 * kConsumerWarps + warp] = pkk;
                    part[2 * kConsumerWarps + warp] = pqk;
                }
            }
            // every consumer learns whether any consumer's wait ran out
            if (consumers_sync_or(!got)) {
                if (t == 0) {
                    report(p.err, GDN_DEVERR_TIMEOUT);
                    atomicExch(&abort_flag, 1);
                }
                break;
            }

            if (live) {
                // ---- norms and gates --------------------------------------------
                float qq = 0.f, kk = 0.f, qk = 0.f;
                constexpr int kRedWarps = (DK + 31) / 32;
#pragma unroll
                for (int wi = 0; wi < kRedWarps; ++wi) {
                    qq += part[0 * kConsumerWarps + wi];
                    kk += part[1 * kConsumerWarps + wi];
                    qk += part[2 * kConsumerWarps + wi];
                }
                const float inv_q = __fdiv_rn(1.0f, sqrtf(qq + kL2Eps)) * rsqrtf((float)DK);
                const float inv_k = __fdiv_rn(1.0f, sqrtf(kk + kL2Eps));
                const float kappa = qk * inv_q * inv_k;
                const float alpha = m.alpha;
                const float beta = m.beta;

                // ---- the state rows ---------------------------------------------
                // every lane runs the reductions (the shuffles need the whole
                // warp); only rows inside the chunk are stored
                const int row = warp * G::RPW + lrow;
                {
                    float4 kh[4], qh[4], sv[4];
                    const float *srow = reinterpret_cast<const float *>(st + L::STATE) + row * DK + 4 * lcol;
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        const int j = 4 * (lcol + G::LPR * mm);
                        const float4 kr = *reinterpret_cast<const float4 *>(&kn[j]);
                        const float4 qr = *reinterpret_cast<const float4 *>(&qn[j]);
                        kh[mm] = make_float4(kr.x * inv_k, kr.y * inv_k, kr.z * inv_k, kr.w * inv_k);
                        qh[mm] = make_float4(qr.x * inv_q, qr.y * inv_q, qr.z * inv_q, qr.w * inv_q);
                        sv[mm] = *reinterpret_cast<const float4 *>(srow + 4 * G::LPR * mm);
                    }
                    float u = 0.f, wd = 0.f;
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        u = __fmaf_rn(sv[mm].x, kh[mm].x, u);
                        u = __fmaf_rn(sv[mm].y, kh[mm].y, u);
                        u = __fmaf_rn(sv[mm].z, kh[mm].z, u);
                        u = __fmaf_rn(sv[mm].w, kh[mm].w, u);
                        wd = __fmaf_rn(sv[mm].x, qh[mm].x, wd);
                        wd = __fmaf_rn(sv[mm].y, qh[mm].y, wd);
                        wd = __fmaf_rn(sv[mm].z, qh[mm].z, wd);
                        wd = __fmaf_rn(sv[mm].w, qh[mm].w, wd);
                    }
#pragma unroll
                    for (int off = G::LPR / 2; off >= 1; off >>= 1) {
                        u += __shfl_xor_sync(0xffffffffu, u, off, G::LPR);
                        wd += __shfl_xor_sync(0xffffffffu, wd, off, G::LPR);
                    }
                    if (row < m.rows) {
                        const float vi = vn[row];
                        const float c = beta * __fmaf_rn(-alpha, u, vi);
                        const float o = __fmaf_rn(c, kappa, alpha * wd);
                        float *dst = p.pool +
                                     (((size_t)m.ws * p.hv + m.h) * p.dv + (size_t)m.chunk * RB + row) * DK +
                                     4 * lcol;
#pragma unroll
                        for (int mm = 0; mm < 4; ++mm) {
                            float4 nv;
                            nv.x = __fmaf_rn(c, kh[mm].x, alpha * sv[mm].x);
                            nv.y = __fmaf_rn(c, kh[mm].y, alpha * sv[mm].y);
                            nv.z = __fmaf_rn(c, kh[mm].z, alpha * sv[mm].z);
                            nv.w = __fmaf_rn(c, kh[mm].w, alpha * sv[mm].w);
                            st_state(dst + 4 * G::LPR * mm, nv);
                        }
                        if (lcol == 0)
                            out[row] = from_f<T>(o);
                    }
                }
            } else if (got) {
                // padding or bad row: zero outputs, no slot touched
                if (t < m.rows)
                    out[t] = from_f<T>(0.f);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty_bar(s));
            if (t == 0)
                consumed_n = k + 1;
        }
    }

    // A CTA whose waits ran out leaves no copy in flight: the producer waits
    // (bounded) for every stage it filled that was not consumed.
    asm volatile("barrier.sync 0;" ::: "memory"); // the producer warp arrives divergently
    if (abort_flag && tid == kConsumers) {
        for (int k = consumed_n; k < issued_n; ++k)
            mbar_wait(full_bar((int)(k % nst)), (uint32_t)((k / nst) & 1));
    }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
int g_num_sms[64] = {};

int num_sms()
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64)
        dev = 0;
    if (!g_num_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_num_sms[dev] = n > 0 ? n : 1;
    }
    return g_num_sms[dev];
}

template <typename T, int DK, bool LAYER, int W>
cudaError_t launch_stream(const StepArgs &a, bool coarse, cudaStream_t s)
{
    using L = Stage<T, DK, LAYER, W>;
    constexpr int RB = Geo<DK>::RB;
    Sched sc;
    sc.hv = a.hv;
    sc.group = a.hv / a.hk;
    sc.chunks = (a.dv + RB - 1) / RB;
    sc.coarse = coarse ? 1 : 0;
    sc.per_unit = coarse ? sc.group * sc.chunks : 1;
    const long long items = (long long)a.rows * a.hv * sc.chunks;
    if (items > (1ll << 30))
        return cudaErrorInvalidValue;
    sc.n_units = (int)(items / sc.per_unit);
    if (sc.n_units == 0)
        return cudaSuccess;
    // two CTAs per SM, each with as many stages as fit (at most 8)
    const int max_smem = (227 * 1024) / kCtasPerSm - 2048;
    int nst = max_smem / L::BYTES;
    nst = nst > 8 ? 8 : nst;
    if (nst < 2)
        return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)nst * L::BYTES;
    auto kern = gdn_stream_kernel<T, DK, LAYER, W>;
    static unsigned long long configured = 0; // one bit per device, per instantiation
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured |= bit;
    }
    const int slots = kCtasPerSm * num_sms();
    const int grid = (int)(sc.n_units < slots ? sc.n_units : slots);
    kern<<<grid, kThreads, smem, s>>>(a, sc, nst);
    return cudaGetLastError();
}

template <typename T, bool LAYER, int W>
cudaError_t dispatch_dk(const StepArgs &a, bool coarse, cudaStream_t s)
{
    switch (a.dk) {
    case 16: return launch_stream<T, 16, LAYER, W>(a, coarse, s);
    case 32: return launch_stream<T, 32, LAYER, W>(a, coarse, s);
    case 64: return launch_stream<T, 64, LAYER, W>(a, coarse, s);
    case 128: return launch_stream<T, 128, LAYER, W>(a, coarse, s);
    case 256: return launch_stream<T, 256, LAYER, W>(a, coarse, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

bool step_shape_supported(int dk, int dv)
{
    return (dk == 16 || dk == 32 || dk == 64 || dk == 128 || dk == 256) && dv >= 8 && dv <= 512 &&
           dv % 8 == 0;
}

bool layer_shape_supported(int dk, int dv, int group, bool in_place)
{
    (void)in_place;
    return step_shape_supported(dk, dv) && group >= 1;
}

cudaError_t launch_gdn_step(const StepArgs &a, int dtype, cudaStream_t s)
{
    if (dtype == GDN_BF16)
        return dispatch_dk<__nv_bfloat16, false, 2>(a, false, s);
    return dispatch_dk<float, false, 2>(a, false, s);
}

cudaError_t launch_gdn_layer(const StepArgs &a, int dtype, cudaStream_t s)
{
    const bool coarse = a.in_place != 0;
    switch (a.width) {
    case 2: return dtype == GDN_BF16 ? dispatch_dk<__nv_bfloat16, true, 2>(a, coarse, s) : dispatch_dk<float, true, 2>(a, coarse, s);
    case 3: return dtype == GDN_BF16 ? dispatch_dk<__nv_bfloat16, true, 3>(a, coarse, s) : dispatch_dk<float, true, 3>(a, coarse, s);
    case 4: return dtype == GDN_BF16 ? dispatch_dk<__nv_bfloat16, true, 4>(a, coarse, s) : dispatch_dk<float, true, 4>(a, coarse, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gdn
