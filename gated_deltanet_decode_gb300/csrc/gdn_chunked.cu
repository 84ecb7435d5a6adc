// The gated delta rule over many tokens a sequence, regrouped over chunks of
// tokens so that its work runs on the tensor cores (gdn_prefill_chunked).
//
// The pages name a chunked GDN path beside the decode kernel ("mstar PR
// #965", section "Correctness": the mixed wrappers are checked against the
// chunked GDN path; "mstar PR #1127": one GDN prefill kernel on Blackwell)
// and print no formula for it.  This kernel computes the recurrence of
// gdn_prefill,
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t,
// regrouped exactly over chunks of C = 64 tokens.  Write the step as
// S_t = alpha_t S_{t-1} + u_t k_t^T with u_t = beta_t (v_t - alpha_t S_{t-1} k_t).
// Inside a chunk that starts from S_0, let G_t be the running sum of
// log alpha (so S_t = e^{G_t} S_0 + sum_{s<=t} e^{G_t-G_s} u_s k_s^T).  With
// Q, K [C][dk] the normalised q and k and V [C][dv]:
//     A[t][s] = beta_t e^{G_t-G_s} (k_t . k_s)    for s < t, else 0
//     P[t][s] = e^{G_t-G_s} (q_t . k_s)           for s <= t, else 0
//     T       = (I + A)^{-1}                       (u's triangular system)
//     E       = (V^T - (S_0 K^T) diag(e^G)) diag(beta)            [dv][C]
//     U^T     = E T^T                                               [dv][C]
//     O^T     = (S_0 Q^T) diag(e^G) + U^T P^T                       [dv][C]
//     S_C     = e^{G_C} S_0 + (U^T diag(e^{G_C-G})) K
// Every exponent is G_t - G_s with s <= t, or G_t itself, so no factor
// exceeds 1 and none overflows.  Tokens past a sequence's end pad the last
// chunk with zero q, k, v and beta and a zero log-gate, which leaves every
// real token's result unchanged.
//
// This file runs fp32 activations; bf16 activations (exact in bf16, so q
// and k need no split) run the tcgen05 kernel of gdn_chunked_tc.cu, which
// keeps the state in tensor memory.
//
// Layout of the work: one CTA per (sequence, value head), 8 warps.  Warp w
// holds state rows 16w..16w+15 (every dk column) in its MMA accumulators for
// the whole sequence, so the state is read once and written once.  Per chunk
// the CTA first loads the chunk's inputs (every load in flight before any is
// used) and builds, in shared memory, the normalised Q and K, the gates,
// A, P and T (T on the CUDA cores in fp32: 16x16 diagonal blocks by forward
// substitution, then the blocks below them); then each warp forms the
// products above for its own rows, and writes its outputs.
//
// Precision: the products run as mma.sync m16n8k16 bf16 with fp32
// accumulation, each fp32 operand split into a bf16 head and a bf16 tail
// (x = hi + lo to about 2^-17 relative); a product sums hi*hi, hi*lo and
// lo*hi, so it carries about 1e-5 relative error instead of bf16's 4e-3.
// The result agrees with the token-serial gdn_prefill within the chained
// state tolerance, not bit for bit.
//
// Sequences, slots and errors follow gdn_prefill exactly: padding (read
// slot 0) and bad sequences zero their outputs and touch no slot, a bad one
// sets the device error word, an empty real sequence moves its state to the
// write slot unchanged.
#include <atomic>

#include "gdn_chunk_common.cuh"
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int CWARPS = 8;        // each holds 16 state rows
constexpr int CTHREADS = CWARPS * 32;
constexpr int LDK = CD + 8;      // row stride (bf16) of [token][dk] tiles: 8 rows hit distinct banks
constexpr int LDT = CK + 8;      // row stride (bf16) of [token][token] tiles
constexpr int LDV = CD + 4;      // row stride (fp32) of the [token][dv] tile

// Shared-memory layout, byte offsets (all 16-byte aligned).
struct CS {
    static constexpr int TOK = CK * LDK * 2;     // one bf16 [CK][LDK] tile
    static constexpr int SQ = CK * LDT * 2;      // one bf16 [CK][LDT] tile
    static constexpr int QH = 0;                 // q head / tail
    static constexpr int QL = QH + TOK;
    static constexpr int KH = QL + TOK;          // k head / tail
    static constexpr int KL = KH + TOK;
    static constexpr int PH = KL + TOK;          // P head / tail [t][s]
    static constexpr int PL = PH + SQ;
    static constexpr int TH = PL + SQ;           // T head / tail [t][s]
    static constexpr int TL = TH + SQ;
    static constexpr int AF = TL + SQ;           // fp32 A [t][s]; its upper blocks hold scratch
    static constexpr int XF = AF + CK * LDF * 4; // fp32 T [t][s]
    static constexpr int VO = XF + CK * LDF * 4; // fp32 [t][dv]: V in, then each warp's outputs
    // gates, two sets (a chunk's and the next one's), each fp32
    // [G (running log-gate) | beta | e^{G_t} | e^{G_C - G_t}] x [CK]
    static constexpr int GATES = VO + CK * LDV * 4;
    static constexpr int BYTES = GATES + 2 * 4 * CK * 4;
};
static_assert(CS::BYTES <= 227 * 1024, "shared memory");
static_assert(CS::AF % 16 == 0 && CS::VO % 16 == 0 && (LDV * 4) % 16 == 0, "alignment");


template <typename TA>
__global__ void __launch_bounds__(CTHREADS, 1) gdn_chunked_kernel(const PrefillArgs p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    bf16 *const QH = reinterpret_cast<bf16 *>(smem + CS::QH);
    bf16 *const QL = reinterpret_cast<bf16 *>(smem + CS::QL);
    bf16 *const KH = reinterpret_cast<bf16 *>(smem + CS::KH);
    bf16 *const KL = reinterpret_cast<bf16 *>(smem + CS::KL);
    bf16 *const PH = reinterpret_cast<bf16 *>(smem + CS::PH);
    bf16 *const PL = reinterpret_cast<bf16 *>(smem + CS::PL);
    bf16 *const TH = reinterpret_cast<bf16 *>(smem + CS::TH);
    bf16 *const TL = reinterpret_cast<bf16 *>(smem + CS::TL);
    float *const AF = reinterpret_cast<float *>(smem + CS::AF);
    float *const XF = reinterpret_cast<float *>(smem + CS::XF);
    float *const VO = reinterpret_cast<float *>(smem + CS::VO);
    float *const GATES = reinterpret_cast<float *>(smem + CS::GATES);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
    const int seq = blockIdx.x / p.hv, h = blockIdx.x - seq * p.hv;
    const int hq = h / (p.hv / p.hk);
    wait_prior_grid();

    const int t0 = p.cu_seqlens[seq], t1 = p.cu_seqlens[seq + 1];
    const bool range_ok = t0 >= 0 && t1 >= t0 && t1 <= p.total_tokens;
    const int rs = p.read_slot[seq];
    const bool in_place = p.write_slot == nullptr;
    const int ws = in_place ? rs : p.write_slot[seq];
    const int cls = range_ok ? classify_row(rs, ws, p.num_slots, in_place) : -1;
    TA *const out = reinterpret_cast<TA *>(p.out);
    const size_t out_tok = (size_t)p.hv * CD;
    if (cls != 1) {
        // padding or bad: zero outputs (when the token range is sane), no slot touched
        if (cls < 0 && h == 0 && tid == 0)
            report(p.err, GDN_DEVERR_BAD_SLOT);
        if (range_ok) {
            const long long n_out = (long long)(t1 - t0) * CD;
            for (long long e = tid; e < n_out; e += CTHREADS)
                out[(size_t)(t0 + e / CD) * out_tok + (size_t)h * CD + (size_t)(e % CD)] = from_f<TA>(0.f);
        }
        return;
    }

    // the state: rows 16w + g and 16w + g + 8 of this warp, columns 8j + 2c, +1
    const size_t slot_floats = (size_t)p.hv * CD * CD;
    const size_t head_off = (size_t)h * CD * CD;
    float sacc[16][4];
    {
        const float *S0 = p.pool + (size_t)rs * slot_floats + head_off + (size_t)(16 * warp + g) * CD + 2 * c;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 x = *reinterpret_cast<const float2 *>(S0 + 8 * j);
            const float2 y = *reinterpret_cast<const float2 *>(S0 + 8 * CD + 8 * j);
            sacc[j][0] = x.x, sacc[j][1] = x.y, sacc[j][2] = y.x, sacc[j][3] = y.y;
        }
    }
    // P's blocks above the diagonal are never computed: zero both halves once
    for (int e = tid; e < 2 * CS::SQ / 4; e += CTHREADS)
        reinterpret_cast<uint32_t *>(PH)[e] = 0u;

    const float rate = expf(p.A_log[h]);
    const float dtb = p.dt_bias[h];
    const float qscale = 1.0f / sqrtf((float)CD);
    const TA *const qg = reinterpret_cast<const TA *>(p.q);
    const TA *const kg = reinterpret_cast<const TA *>(p.k);
    const TA *const vg = reinterpret_cast<const TA *>(p.v);
    const TA *const ag = reinterpret_cast<const TA *>(p.a);
    const TA *const bg = reinterpret_cast<const TA *>(p.b);
    const int L = t1 - t0;

    // the gate inputs of the chunk starting at cn: warp 2, tokens lane and lane + 32
    TA ra[2], rb[2];
    auto gates_in = [&](int cn) {
        const int nn = min(CK, L - cn);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int tt = lane + 32 * i;
            if (tt < nn) {
                const size_t idx = (size_t)(t0 + cn + tt) * p.hv + h;
                ra[i] = ag[idx], rb[i] = bg[idx];
            }
        }
    };
    // the gates of the chunk starting at cn from ra, rb (warp 2): log alpha,
    // beta, running sums (zero past the chunk's tokens), into set `set`
    auto gates = [&](int cn, int set) {
        chunk_gates(GATES + set * 4 * CK, ra, rb, min(CK, L - cn), rate, dtb, lane);
    };
    if (L > 0) {
        if (warp == 2) {
            gates_in(0);
            gates(0, 0);
        }
    }

#pragma unroll 1
    for (int c0 = 0; c0 < L; c0 += CK) {
        const int n = min(CK, L - c0);
        const int set = (c0 / CK) & 1;
        const float *const GG = GATES + set * 4 * CK; // this chunk's gates
        const float *const BE = GG + CK;
        const float *const EG = GG + 2 * CK;
        const float *const EC = GG + 3 * CK;
        const bool more = c0 + CK < L;
        __syncthreads(); // every warp is done with the previous chunk's tiles

        // ---- the chunk's inputs, every load in flight before any is used:
        // q, k, v: 8 tokens a warp (token warp + 8i), 4 channels a lane ----
        constexpr int TPW = CK / CWARPS;
        Raw4<TA> rq[TPW], rk[TPW], rv[TPW];
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
            const int tt = warp + CWARPS * i;
            if (tt < n) {
                const size_t tok = (size_t)(t0 + c0 + tt);
                rq[i] = ldraw<TA>(qg + (tok * p.hk + hq) * CD + 4 * lane);
                rk[i] = ldraw<TA>(kg + (tok * p.hk + hq) * CD + 4 * lane);
                rv[i] = ldraw<TA>(vg + (tok * p.hv + h) * CD + 4 * lane);
            } else {
                rq[i] = raw_zero<TA>(), rk[i] = raw_zero<TA>(), rv[i] = raw_zero<TA>();
            }
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
            const int tt = warp + CWARPS * i;
            float qv[4], kv[4], vv[4];
            unpack(qv, rq[i]), unpack(kv, rk[i]), unpack(vv, rv[i]);
            float sq = qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3];
            float sk = kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3];
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float iq = qscale * rsqrtf(sq + kEps), ik = rsqrtf(sk + kEps);
            uint32_t h0, l0, h1, l1;
            split2(qv[0] * iq, qv[1] * iq, h0, l0);
            split2(qv[2] * iq, qv[3] * iq, h1, l1);
            *reinterpret_cast<uint2 *>(QH + tt * LDK + 4 * lane) = make_uint2(h0, h1);
            *reinterpret_cast<uint2 *>(QL + tt * LDK + 4 * lane) = make_uint2(l0, l1);
            split2(kv[0] * ik, kv[1] * ik, h0, l0);
            split2(kv[2] * ik, kv[3] * ik, h1, l1);
            *reinterpret_cast<uint2 *>(KH + tt * LDK + 4 * lane) = make_uint2(h0, h1);
            *reinterpret_cast<uint2 *>(KL + tt * LDK + 4 * lane) = make_uint2(l0, l1);
            *reinterpret_cast<float4 *>(VO + tt * LDV + 4 * lane) = make_float4(vv[0], vv[1], vv[2], vv[3]);
        }
        __syncthreads();
        // the next chunk's gate inputs travel while this one computes
        if (more && warp == 2)
            gates_in(c0 + CK);

        // ---- K K^T -> A and Q K^T -> P: the 8-column tiles of their lower
        // 16x16 blocks (10 blocks x 2 tiles x 2 products = 40), 5 a warp,
        // their accumulation chains interleaved ----
        {
            constexpr int NT = 40 / CWARPS;
            float acc[NT][4];
            int mrow[NT], ncol[NT];
            bool isq[NT];
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const int tau = warp + CWARPS * i;
                isq[i] = tau >= 20;
                const int idx = isq[i] ? tau - 20 : tau;
                const int blk = idx >> 1;
                const int mb = blk >= 6 ? 3 : blk >= 3 ? 2 : blk >= 1 ? 1 : 0;
                mrow[i] = 16 * mb;
                ncol[i] = 16 * (blk - mb * (mb + 1) / 2) + 8 * (idx & 1);
                acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
            }
#pragma unroll
            for (int kb = 0; kb < CD / 16; ++kb) {
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    uint32_t ah[4], al[4], bh0, bh1, bl0, bl1;
                    lda(ah, isq[i] ? QH : KH, LDK, mrow[i], 16 * kb, g, c);
                    ldb(bh0, bh1, KH, LDK, ncol[i], 16 * kb, g, c);
                    lda(al, isq[i] ? QL : KL, LDK, mrow[i], 16 * kb, g, c);
                    ldb(bl0, bl1, KL, LDK, ncol[i], 16 * kb, g, c);
                    mma3(acc[i], ah, al, bh0, bh1, bl0, bl1);
                }
            }
#pragma unroll
            for (int i = 0; i < NT; ++i) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int t = mrow[i] + g + 8 * hr;
                    const int s = ncol[i] + 2 * c;
                    const float x = acc[i][2 * hr], y = acc[i][2 * hr + 1];
                    const float gt = GG[t];
                    if (!isq[i]) {
                        const float bt = BE[t];
                        *reinterpret_cast<float2 *>(AF + t * LDF + s) =
                            make_float2(s < t ? bt * expf(gt - GG[s]) * x : 0.f,
                                        s + 1 < t ? bt * expf(gt - GG[s + 1]) * y : 0.f);
                    } else {
                        const float px = s <= t ? expf(gt - GG[s]) * x : 0.f;
                        const float py = s + 1 <= t ? expf(gt - GG[s + 1]) * y : 0.f;
                        uint32_t hh, ll;
                        split2(px, py, hh, ll);
                        *reinterpret_cast<uint32_t *>(PH + t * LDT + s) = hh;
                        *reinterpret_cast<uint32_t *>(PL + t * LDT + s) = ll;
                    }
                }
            }
        }
        __syncthreads();

        // ---- T = (I + A)^{-1}, fp32: diagonal blocks, then the blocks below ----
        if (tid < CK)
            t_diagonal(AF, XF, tid);
        else if (more && warp == 2)
            gates(c0 + CK, set ^ 1); // meanwhile: the next chunk's gates
        __syncthreads();
        t_below_diagonal(AF, XF, warp, g, c);
        // T's lower triangle, split (above it: zero)
        for (int e = tid; e < CK * CK / 2; e += CTHREADS) {
            const int t = e / (CK / 2), s = 2 * (e % (CK / 2));
            const float2 v = *reinterpret_cast<const float2 *>(XF + t * LDF + s);
            const float x = s <= t ? v.x : 0.f;
            const float y = s + 1 <= t ? v.y : 0.f;
            uint32_t hh, ll;
            split2(x, y, hh, ll);
            *reinterpret_cast<uint32_t *>(TH + t * LDT + s) = hh;
            *reinterpret_cast<uint32_t *>(TL + t * LDT + s) = ll;
        }
        __syncthreads();

        // the next chunk's q, k, v travel during this chunk's products (a
        // warp stalled on issuing them leaves the tensor pipe to the other)
        // ---- this warp's rows: Z = S K^T and Y = S Q^T (16 x 64 each) ----
        float z[8][4], y[8][4], u[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                z[nt][e] = 0.f, y[nt][e] = 0.f, u[nt][e] = 0.f;
#pragma unroll
        for (int kb = 0; kb < CD / 16; ++kb) {
            uint32_t ah[4], al[4];
            acc_to_a(ah, al, sacc[2 * kb], sacc[2 * kb + 1]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                uint32_t bh0, bh1, bl0, bl1;
                ldb(bh0, bh1, KH, LDK, 8 * nt, 16 * kb, g, c);
                ldb(bl0, bl1, KL, LDK, 8 * nt, 16 * kb, g, c);
                mma3(z[nt], ah, al, bh0, bh1, bl0, bl1);
                ldb(bh0, bh1, QH, LDK, 8 * nt, 16 * kb, g, c);
                ldb(bl0, bl1, QL, LDK, 8 * nt, 16 * kb, g, c);
                mma3(y[nt], ah, al, bh0, bh1, bl0, bl1);
            }
        }
        // E = (V^T - Z diag(e^G)) diag(beta), in place of Z
        const int rA = 16 * warp + g;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 8 * nt + 2 * c + (e & 1), r = rA + 8 * (e >> 1);
                z[nt][e] = BE[t] * (VO[t * LDV + r] - EG[t] * z[nt][e]);
            }
        // U^T = E T^T
#pragma unroll
        for (int kb = 0; kb < CK / 16; ++kb) {
            uint32_t ah[4], al[4];
            acc_to_a(ah, al, z[2 * kb], z[2 * kb + 1]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                uint32_t bh0, bh1, bl0, bl1;
                ldb(bh0, bh1, TH, LDT, 8 * nt, 16 * kb, g, c);
                ldb(bl0, bl1, TL, LDT, 8 * nt, 16 * kb, g, c);
                mma3(u[nt], ah, al, bh0, bh1, bl0, bl1);
            }
        }
        // O^T = Y diag(e^G) + U^T P^T
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int t = 8 * nt + 2 * c;
            const float e0 = EG[t], e1 = EG[t + 1];
            y[nt][0] *= e0, y[nt][1] *= e1, y[nt][2] *= e0, y[nt][3] *= e1;
        }
#pragma unroll
        for (int kb = 0; kb < CK / 16; ++kb) {
            uint32_t ah[4], al[4];
            acc_to_a(ah, al, u[2 * kb], u[2 * kb + 1]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                uint32_t bh0, bh1, bl0, bl1;
                ldb(bh0, bh1, PH, LDT, 8 * nt, 16 * kb, g, c);
                ldb(bl0, bl1, PL, LDT, 8 * nt, 16 * kb, g, c);
                mma3(y[nt], ah, al, bh0, bh1, bl0, bl1);
            }
        }
        // outputs into this warp's own columns of the V tile (this lane read exactly these)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 8 * nt + 2 * c + (e & 1), r = rA + 8 * (e >> 1);
                VO[t * LDV + r] = y[nt][e];
            }
        // S = e^{G_C} S + (U^T diag(e^{G_C - G})) K
        const float gC = EG[CK - 1];
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sacc[j][e] *= gC;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int t = 8 * nt + 2 * c;
            const float e0 = EC[t], e1 = EC[t + 1];
            u[nt][0] *= e0, u[nt][1] *= e1, u[nt][2] *= e0, u[nt][3] *= e1;
        }
#pragma unroll
        for (int kb = 0; kb < CK / 16; ++kb) {
            uint32_t ah[4], al[4];
            acc_to_a(ah, al, u[2 * kb], u[2 * kb + 1]);
#pragma unroll
            for (int np = 0; np < CD / 16; ++np) {
                uint32_t bh[4], bl[4];
                ldb_trans2(bh, KH, LDK, 16 * kb, 16 * np, lane);
                ldb_trans2(bl, KL, LDK, 16 * kb, 16 * np, lane);
                mma3(sacc[2 * np], ah, al, bh[0], bh[1], bl[0], bl[1]);
                mma3(sacc[2 * np + 1], ah, al, bh[2], bh[3], bl[2], bl[3]);
            }
        }
        __syncwarp();
        // this warp's 16 output columns of each real token: 8 lanes a token, two values a lane
        for (int e = lane; e < n * 8; e += 32) {
            const int t = e >> 3, r = 16 * warp + 2 * (e & 7);
            const float2 v2 = *reinterpret_cast<const float2 *>(VO + t * LDV + r);
            store2<TA>(out + (size_t)(t0 + c0 + t) * out_tok + (size_t)h * CD + r, v2.x, v2.y);
        }
    }

    // the final state, to the write slot (the read slot in place)
    {
        float *Sd = p.pool + (size_t)ws * slot_floats + head_off + (size_t)(16 * warp + g) * CD + 2 * c;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            *reinterpret_cast<float2 *>(Sd + 8 * j) = make_float2(sacc[j][0], sacc[j][1]);
            *reinterpret_cast<float2 *>(Sd + 8 * CD + 8 * j) = make_float2(sacc[j][2], sacc[j][3]);
        }
    }
}

template <typename TA>
cudaError_t launch_chunked_t(const PrefillArgs &a, cudaStream_t s)
{
    const long long ctas = (long long)a.nseq * a.hv;
    if (ctas == 0)
        return cudaSuccess;
    if (ctas > 0x7fffffffll)
        return cudaErrorInvalidValue;
    auto kern = gdn_chunked_kernel<TA>;
    static std::atomic<unsigned long long> configured{0}; // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CS::BYTES);
        if (e != cudaSuccess)
            return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    return launch_pdl(kern, dim3((unsigned)ctas), dim3(CTHREADS), (size_t)CS::BYTES, s, a);
}

} // namespace

bool chunked_shape_supported(int dk, int dv) { return dk == CD && dv == CD; }

cudaError_t launch_gdn_prefill_chunked(const PrefillArgs &a, int dtype, cudaStream_t s)
{
    if (!chunked_shape_supported(a.dk, a.dv))
        return cudaErrorInvalidValue;
    return dtype == GDN_BF16 ? launch_gdn_prefill_chunked_tc(a, s) : launch_chunked_t<float>(a, s);
}

} // namespace gdn
