// gdn_prefill / gdn_verify: the gated delta rule over many tokens a sequence,
// sm_103a.
//
// A prefill is the decode rule applied token after token, keeping the state
// ("mstar PR #1139", section "Why": the rule is the recurrent state update,
// and prefill keeps the state in place); verification keeps the state after
// every token in a slot of its own (section "What changed": speculative
// decoding holds a state per token, so twin slots do not apply to it).
//
// Work item = RB = 4096 / dk value rows of one (sequence, value head): 16 KiB
// of fp32 state, read once into registers (16 floats a lane, the decode
// kernel's geometry) and written once at the end (or once a token when
// verifying).  A persistent grid (two CTAs an SM) splits the items into
// contiguous ranges.  A loader warp bulk-copies the next item's state rows
// into one of two state buffers while the current item's tokens run, and
// streams every token's raw q, k and v chunk through a ring of shared-memory
// stages, with the gates computed 32 tokens at a time; two norm warps,
// taking alternate tokens, turn q and k into fp32 values and form their
// norms and k^ . q^; the 8 consumer warps then only update their state rows.  Every sum is formed
// with the decode kernel's operations in its order (the norm warps play the
// decode kernel's 8 consumer warps lane by lane), so T tokens of a prefill
// equal T decode steps bit for bit.
//
// The rule is sequential in the tokens: an item's work is one token after
// the other; short sequences (verification) are bound by the state traffic,
// which the state prefetch keeps flowing.  (The chunked form,
// which turns runs of tokens into dense products for the tensor cores, is a
// different kernel; this one is exact with respect to the decode step.)
#include <atomic>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_ptx.cuh"

namespace gdn {

namespace {

constexpr int kWarps = 8;                    // consumer warps
constexpr int kConsumerThreads = kWarps * 32;
constexpr int kNormWarps = 2;                // warps that normalise q and k, alternate tokens
constexpr int kLoader = kWarps;              // warp index of the loader
constexpr int kThreads = (kWarps + 1 + kNormWarps) * 32;
constexpr int kStages = 8;                   // token ring depth
constexpr float kL2Eps = 1e-6f;

template <int DK> struct PGeo {
    static_assert(DK >= 16 && DK <= 256 && DK % 16 == 0, "dk");
    static constexpr int LPR = DK / 16;      // lanes per state row
    static constexpr int RPW = 32 / LPR;     // state rows per warp
    static constexpr int RB = RPW * kWarps;  // state rows per CTA (4096 / DK)
};

// One token's raw inputs: q[DK] | k[DK] | v[RB], activation type.
template <typename T, int DK> struct PStage {
    static constexpr int E = sizeof(T);
    static constexpr int QK = 0;
    static constexpr int V = 2 * DK * E;
    static constexpr int BYTES = (V + PGeo<DK>::RB * E + 15) & ~15;
};

template <typename T>
__device__ __forceinline__ float sh_val(const unsigned char *base, int idx)
{
    return to_f(reinterpret_cast<const T *>(base)[idx]);
}
template <typename T>
__device__ __forceinline__ float gl_val(const void *base, size_t idx)
{
    return to_f(reinterpret_cast<const T *>(base)[idx]);
}

// Dynamic shared memory of a CTA: the token ring (raw inputs), the tokens'
// fp32 q|k values, and two state buffers (the next item's state lands while
// the current item's tokens run).
template <typename T, int DK> struct PSmem {
    static constexpr int RB = PGeo<DK>::RB;
    static constexpr int RING = 0;
    static constexpr int QKF = (RING + kStages * PStage<T, DK>::BYTES + 127) & ~127;
    static constexpr int SBUF = (QKF + kStages * 2 * DK * 4 + 127) & ~127;
    static constexpr int SBUF_BYTES = RB * DK * 4;
    static constexpr int BYTES = SBUF + 2 * SBUF_BYTES;
};

// What the loader learned about an item (a sequence, value head and row
// block), handed to the other warps through a double-buffered table.
struct ItemMeta {
    int cls;  // 1 real, 0 padding, -1 bad
    int t0, n; // the sequence's first token and token count
    int rs, ws, h, chunk, rows;
};

template <typename T, int DK>
__global__ void __launch_bounds__(kThreads, 2) gdn_prefill_kernel(const PrefillArgs p, int n_items)
{
    using G = PGeo<DK>;
    using L = PStage<T, DK>;
    using M = PSmem<T, DK>;
    constexpr int RB = G::RB;
    constexpr int E = L::E;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem + M::RING;
    __shared__ __align__(8) unsigned long long bars[3 * kStages + 4]; // full, ready, empty; item full, empty
    __shared__ ItemMeta imeta[2];
    __shared__ float norm_q[kStages], norm_k[kStages], kap[kStages];
    __shared__ float gate_a[kStages], gate_b[kStages];
    __shared__ float tab_a[32], tab_b[32];
    __shared__ int abort_flag, issued_n, consumed_n, items_issued, items_read;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int chunks = (p.dv + RB - 1) / RB;
    const int group = p.hv / p.hk;
    const bool verify = p.token_slot != nullptr;
    const size_t out_tok = (size_t)p.hv * p.dv;       // output elements a token
    const size_t slot_floats = (size_t)p.hv * p.dv * DK;
    // this CTA's items: a contiguous range, equal to within one
    const int i0 = (int)(((long long)n_items * blockIdx.x) / gridDim.x);
    const int i1 = (int)(((long long)n_items * (blockIdx.x + 1)) / gridDim.x);
    const int n_mine = i1 - i0;
    auto full_bar = [&](int s) { return sm_addr(&bars[s]); };
    auto ready_bar = [&](int s) { return sm_addr(&bars[kStages + s]); };
    auto empty_bar = [&](int s) { return sm_addr(&bars[2 * kStages + s]); };
    auto ifull_bar = [&](int b) { return sm_addr(&bars[3 * kStages + b]); };
    auto iempty_bar = [&](int b) { return sm_addr(&bars[3 * kStages + 2 + b]); };
    auto qkf = [&](int s) { return reinterpret_cast<float *>(smem + M::QKF) + (size_t)s * 2 * DK; };
    auto sbuf = [&](int b) { return reinterpret_cast<float *>(smem + M::SBUF + (size_t)b * M::SBUF_BYTES); };
    auto timeout = [&]() {
        report(p.err, GDN_DEVERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 2);  // copies + gates
            mbar_init(ready_bar(s), 1); // the token's norm warp
            mbar_init(empty_bar(s), kWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(ifull_bar(b), 2); // state copy + metadata
            mbar_init(iempty_bar(b), kWarps + kNormWarps);
        }
        abort_flag = 0;
        issued_n = consumed_n = items_issued = items_read = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    wait_prior_grid();

    if (warp == kLoader) {
        // ============================ loader ============================
        // For each item: its sequence's classification, its metadata and (for
        // a real sequence) the bulk copy of its state rows into a state
        // buffer; then its tokens' raw q, k and v chunk, streamed into the
        // token ring with their gates (computed 32 tokens at a time).
        const unsigned char *qp = reinterpret_cast<const unsigned char *>(p.q);
        const unsigned char *kp = reinterpret_cast<const unsigned char *>(p.k);
        const unsigned char *vp = reinterpret_cast<const unsigned char *>(p.v);
        bool stop = false;
        int K = 0; // tokens streamed so far (the ring's running index)
        for (int li = 0; li < n_mine && !stop; ++li) {
            const int item = i0 + li, ib = li & 1;
            const int chunk = item % chunks;
            const int rh = item / chunks;
            const int h = rh % p.hv, r = rh / p.hv;
            const int t0 = p.cu_seqlens[r], t1 = p.cu_seqlens[r + 1];
            const int rs = p.read_slot[r];
            const bool in_place = p.write_slot == nullptr || verify;
            const int ws = in_place ? rs : p.write_slot[r];
            int cls;
            if (t0 < 0 || t1 < t0 || t1 > p.total_tokens)
                cls = -1;
            else
                cls = classify_row(rs, ws, p.num_slots, in_place);
            if (cls == 1 && verify) {
                bool bad = false;
                for (int t = t0 + lane; t < t1; t += 32) {
                    const int s = p.token_slot[t];
                    bad |= s <= 0 || s >= p.num_slots || s == rs;
                }
                if (__any_sync(0xffffffffu, bad))
                    cls = -1;
            }
            const int rows = min(RB, p.dv - chunk * RB);
            const int n = cls == 1 ? t1 - t0 : 0;
            if (lane == 0) {
                if (cls < 0 && h == 0 && chunk == 0)
                    report(p.err, GDN_DEVERR_BAD_SLOT);
                if (!mbar_wait(iempty_bar(ib), (uint32_t)((li >> 1) & 1) ^ 1u)) {
                    timeout();
                    stop = true;
                } else {
                    ItemMeta m;
                    m.cls = cls;
                    m.t0 = t0;
                    m.n = t1 - t0;
                    m.rs = rs;
                    m.ws = ws;
                    m.h = h;
                    m.chunk = chunk;
                    m.rows = rows;
                    imeta[ib] = m;
                    const uint32_t fb = ifull_bar(ib);
                    if (cls == 1) {
                        mbar_arrive_tx(fb, (uint32_t)(rows * DK * 4));
                        bulk_load(sm_addr(sbuf(ib)),
                                  p.pool + (size_t)rs * slot_floats + ((size_t)h * p.dv + (size_t)chunk * RB) * DK,
                                  (uint32_t)(rows * DK * 4), fb);
                    } else {
                        mbar_arrive(fb);
                    }
                    mbar_arrive(fb);
                    items_issued = li + 1;
                }
            }
            stop = __shfl_sync(0xffffffffu, stop, 0);
            const float al = p.A_log[h], dt = p.dt_bias[h];
            const int g = h / group;
            for (int base = 0; base < n && !stop; base += 32) {
                const int kk = base + lane;
                float ga = 0.f, gb = 0.f;
                if (kk < n) {
                    const size_t t = (size_t)(t0 + kk);
                    ga = gate_alpha(al, gl_val<T>(p.a, t * p.hv + h), dt);
                    gb = gate_beta(gl_val<T>(p.b, t * p.hv + h));
                }
                tab_a[lane] = ga;
                tab_b[lane] = gb;
                __syncwarp();
                if (lane == 0) {
                    const int nb = min(32, n - base);
                    for (int j = 0; j < nb; ++j) {
                        const int k = K + base + j, s = k % kStages;
                        if (!mbar_wait(empty_bar(s), (uint32_t)((k / kStages) & 1) ^ 1u)) {
                            timeout();
                            stop = true;
                            break;
                        }
                        if (*(volatile int *)&abort_flag) {
                            stop = true;
                            break;
                        }
                        const size_t t = (size_t)(t0 + base + j);
                        unsigned char *st = ring + (size_t)s * L::BYTES;
                        const uint32_t fb = full_bar(s);
                        mbar_arrive_tx(fb, (uint32_t)((2 * DK + rows) * E));
                        bulk_load(sm_addr(st + L::QK), qp + (t * p.hk + g) * DK * E, DK * E, fb);
                        bulk_load(sm_addr(st + L::QK + DK * E), kp + (t * p.hk + g) * DK * E, DK * E, fb);
                        bulk_load(sm_addr(st + L::V), vp + ((t * p.hv + h) * p.dv + (size_t)chunk * RB) * E,
                                  (uint32_t)(rows * E), fb);
                        gate_a[s] = tab_a[j];
                        gate_b[s] = tab_b[j];
                        mbar_arrive(fb);
                        issued_n = k + 1;
                    }
                }
                stop = __shfl_sync(0xffffffffu, stop, 0);
                __syncwarp();
            }
            K += n;
        }
    } else if (warp > kLoader) {
        // ========================== norm warps ==========================
        // Token k of the ring belongs to norm warp k % kNormWarps.  Lane l
        // plays thread 32w + l of the decode kernel's consumer warp w, for
        // every w: the same channels, the same fma chains, the same
        // butterflies, the same order of the per-warp sums, so the norms and
        // k^ . q^ are the decode kernel's to the bit.
        const int nw = warp - kLoader - 1;
        int K = 0;
        for (int li = 0; li < n_mine; ++li) {
            const int ib = li & 1;
            if (!mbar_wait(ifull_bar(ib), (uint32_t)((li >> 1) & 1))) {
                timeout();
                break;
            }
            const int n = imeta[ib].cls == 1 ? imeta[ib].n : 0;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(iempty_bar(ib));
            bool ok = true;
            for (int k = K + ((nw - K % kNormWarps + kNormWarps) % kNormWarps); k < K + n; k += kNormWarps) {
                const int s = k % kStages;
                if (!mbar_wait(full_bar(s), (uint32_t)((k / kStages) & 1))) {
                    timeout();
                    ok = false;
                    break;
                }
                const unsigned char *st = ring + (size_t)s * L::BYTES;
                float *qf = qkf(s);
                float pq[kWarps], pk[kWarps];
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    float a = 0.f, b = 0.f;
#pragma unroll
                    for (int c0 = 32 * w; c0 < 2 * DK; c0 += kConsumerThreads) {
                        const int c = c0 + lane;
                        const float val = sh_val<T>(st + L::QK, c);
                        qf[c] = val;
                        if (c < DK)
                            a = __fmaf_rn(val, val, a);
                        else
                            b = __fmaf_rn(val, val, b);
                    }
                    pq[w] = a;
                    pk[w] = b;
                }
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    // a warp without q (or k) channels sums exact zeros: skip its butterfly
                    if (32 * w < DK) {
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1)
                            pq[w] += __shfl_xor_sync(0xffffffffu, pq[w], off);
                    }
                    if ((32 * w < 2 * DK && 32 * w + 31 >= DK) || 32 * w + kConsumerThreads < 2 * DK) {
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1)
                            pk[w] += __shfl_xor_sync(0xffffffffu, pk[w], off);
                    }
                }
                float qq = 0.f, kk2 = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    qq += pq[w];
                    kk2 += pk[w];
                }
                const float inv_q = __fdiv_rn(1.0f, sqrtf(qq + kL2Eps)) * rsqrtf((float)DK);
                const float inv_k = __fdiv_rn(1.0f, sqrtf(kk2 + kL2Eps));
                __syncwarp();
                float pqk = 0.f;
                for (int i = lane; i < DK; i += 32)
                    pqk = __fmaf_rn(qf[i], qf[DK + i], pqk);
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
                    pqk += __shfl_xor_sync(0xffffffffu, pqk, off);
                if (lane == 0) {
                    norm_q[s] = inv_q;
                    norm_k[s] = inv_k;
                    kap[s] = pqk * inv_q * inv_k;
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(ready_bar(s));
            }
            if (!ok)
                break;
            K += n;
        }
    } else {
        // =========================== consumers ==========================
        const int lrow = lane / G::LPR, lcol = lane % G::LPR;
        const int t = tid; // consumer index 0..255
        const int row = warp * G::RPW + lrow;
        int K = 0;
        bool ok = true;
        for (int li = 0; li < n_mine && ok; ++li) {
            const int ib = li & 1;
            if (!mbar_wait(ifull_bar(ib), (uint32_t)((li >> 1) & 1))) {
                timeout();
                break;
            }
            const ItemMeta m = imeta[ib];
            const bool live_row = row < m.rows;
            float4 sv[4];
            if (m.cls == 1) {
                // the item's state rows, landed in the state buffer
                const float *sb = sbuf(ib) + row * DK + 4 * lcol;
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    sv[mm] = live_row ? *reinterpret_cast<const float4 *>(sb + 4 * G::LPR * mm)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(iempty_bar(ib));
            if (t == 0)
                items_read = li + 1;
            T *outb = reinterpret_cast<T *>(p.out) + (size_t)m.h * p.dv + (size_t)m.chunk * RB;
            if (m.cls != 1) {
                // padding or bad: zero outputs (when the token range is sane), no slot touched
                if (m.t0 >= 0 && m.n >= 0 && m.t0 + m.n <= p.total_tokens) {
                    const long long n_out = (long long)m.n * m.rows;
                    for (long long e = t; e < n_out; e += kConsumerThreads)
                        outb[(size_t)(m.t0 + e / m.rows) * out_tok + (size_t)(e % m.rows)] = from_f<T>(0.f);
                }
                continue;
            }
            const size_t row_off = ((size_t)m.h * p.dv + (size_t)m.chunk * RB + row) * DK + 4 * lcol;
            for (int k = K; k < K + m.n; ++k) {
                const int s = k % kStages;
                if (!mbar_wait(ready_bar(s), (uint32_t)((k / kStages) & 1))) {
                    timeout();
                    ok = false;
                    break;
                }
                const unsigned char *st = ring + (size_t)s * L::BYTES;
                const float *qk = qkf(s);
                const float inv_q = norm_q[s], inv_k = norm_k[s], kappa = kap[s];
                const float alpha = gate_a[s], beta = gate_b[s];
                const float vi = live_row ? sh_val<T>(st + L::V, row) : 0.f;
                float4 kh[4], qh[4];
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    const int j = 4 * (lcol + G::LPR * mm);
                    qh[mm] = *reinterpret_cast<const float4 *>(&qk[j]);
                    kh[mm] = *reinterpret_cast<const float4 *>(&qk[DK + j]);
                }
                // everything this warp needs from the stage is in registers
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty_bar(s));
                float2 u2 = make_float2(0.f, 0.f), w2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    u2 = fma2(make_float2(sv[mm].x, sv[mm].y), make_float2(kh[mm].x, kh[mm].y), u2);
                    u2 = fma2(make_float2(sv[mm].z, sv[mm].w), make_float2(kh[mm].z, kh[mm].w), u2);
                    w2 = fma2(make_float2(sv[mm].x, sv[mm].y), make_float2(qh[mm].x, qh[mm].y), w2);
                    w2 = fma2(make_float2(sv[mm].z, sv[mm].w), make_float2(qh[mm].z, qh[mm].w), w2);
                }
                float u = u2.x + u2.y, wd = w2.x + w2.y;
#pragma unroll
                for (int off = G::LPR / 2; off >= 1; off >>= 1) {
                    u += __shfl_xor_sync(0xffffffffu, u, off);
                    wd += __shfl_xor_sync(0xffffffffu, wd, off);
                }
                u *= inv_k;  // S . k^
                wd *= inv_q; // S . q^
                if (live_row) {
                    const float c = beta * __fmaf_rn(-alpha, u, vi);
                    const float o = __fmaf_rn(c, kappa, alpha * wd);
                    const float ck = c * inv_k;
                    const float2 a2 = make_float2(alpha, alpha), c2 = make_float2(ck, ck);
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        const float2 lo = fma2(c2, make_float2(kh[mm].x, kh[mm].y),
                                               mul2(a2, make_float2(sv[mm].x, sv[mm].y)));
                        const float2 hi = fma2(c2, make_float2(kh[mm].z, kh[mm].w),
                                               mul2(a2, make_float2(sv[mm].z, sv[mm].w)));
                        sv[mm] = make_float4(lo.x, lo.y, hi.x, hi.y);
                    }
                    const size_t tok = (size_t)(m.t0 + (k - K));
                    if (lcol == 0)
                        outb[tok * out_tok + row] = from_f<T>(o);
                    if (verify) {
                        float *dst = p.pool + (size_t)p.token_slot[tok] * slot_floats + row_off;
#pragma unroll
                        for (int mm = 0; mm < 4; ++mm)
                            st_state(dst + 4 * G::LPR * mm, sv[mm]);
                    }
                }
                if (t == 0)
                    consumed_n = k + 1;
            }
            if (ok && !verify && live_row) {
                float *dst = p.pool + (size_t)m.ws * slot_floats + row_off;
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    st_state(dst + 4 * G::LPR * mm, sv[mm]);
            }
            K += m.n;
        }
    }

    // A CTA whose waits ran out leaves no copy in flight: the loader waits
    // (bounded) for every token stage and state buffer it filled that was
    // not consumed.
    asm volatile("barrier.sync 0;" ::: "memory");
    if (abort_flag && tid == kLoader * 32) {
        for (int k = consumed_n; k < issued_n; ++k)
            mbar_wait(full_bar(k % kStages), (uint32_t)((k / kStages) & 1));
        for (int li = items_read; li < items_issued; ++li)
            mbar_wait(ifull_bar(li & 1), (uint32_t)((li >> 1) & 1));
    }
}

template <typename T, int DK>
cudaError_t launch_dk(const PrefillArgs &a, cudaStream_t s)
{
    using M = PSmem<T, DK>;
    constexpr int RB = PGeo<DK>::RB;
    const long long chunks = (a.dv + RB - 1) / RB;
    const long long items = (long long)a.nseq * a.hv * chunks;
    if (items == 0)
        return cudaSuccess;
    if (items > 0x7fffffffll)
        return cudaErrorInvalidValue;
    auto kern = gdn_prefill_kernel<T, DK>;
    static std::atomic<unsigned long long> configured{0}; // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, M::BYTES);
        if (e != cudaSuccess)
            return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long slots = 2ll * (sms > 0 ? sms : 1);
    const int grid = (int)(items < slots ? items : slots);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)M::BYTES, s, a, (int)items);
}

template <typename T>
cudaError_t launch_t(const PrefillArgs &a, cudaStream_t s)
{
    switch (a.dk) {
    case 16: return launch_dk<T, 16>(a, s);
    case 32: return launch_dk<T, 32>(a, s);
    case 64: return launch_dk<T, 64>(a, s);
    case 128: return launch_dk<T, 128>(a, s);
    case 256: return launch_dk<T, 256>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

cudaError_t launch_gdn_prefill(const PrefillArgs &a, int dtype, cudaStream_t s)
{
    return dtype == GDN_BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

} // namespace gdn
