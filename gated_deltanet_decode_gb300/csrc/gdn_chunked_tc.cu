// The chunked gated delta rule with the state in tensor memory: the
// tcgen05 form of gdn_prefill_chunked for bf16 activations.  The pages name
// the chunked GDN path, check the mixed step against it ("mstar PR #965",
// "Correctness") and run prefill as one GDN kernel ("mstar PR #1127"); they
// print no formula, so the regrouping below is derived from the recurrence.
//
// The operation, the regrouping over chunks of 64 tokens and the split
// products are those of gdn_chunked.cu (whose header states the algebra):
// per chunk A, P and T = (I + A)^{-1}, then with S_0 the state before it
//     Z = S_0 K^T, Y = S_0 Q^T,  E = (V^T - Z diag(e^G ik)) diag(beta),
//     U = E T^T,  O = Y diag(e^G iq) + U P^T,
//     S_C = e^{G_C} S_0 + U diag(e^{G_C-G} ik) K
// (ik, iq: the per-token norm scales of the raw bf16 k and q, which are exact
// operands).
//
// Two kernels.  The prep kernel (one CTA per workspace unit and value head)
// forms every chunk's state-free terms at once -- the gates, the norm scales,
// P and T split into bf16 heads and tails -- into a caller-owned workspace.
// The chunk kernel (one CTA per sequence and value head) then carries the
// state through the chunks in order:
//   * the state S lives in TMEM for the whole sequence (fp32, 128 columns);
//     the products are M = 128 tcgen05.mma with their A operands in TMEM
//     (the bf16 head and tail of S, E, U and U diag(e^{G_C-G} ik)) and their
//     B operands in shared memory: raw K and Q in the 128-byte-swizzled
//     K-major layout a tensor copy writes, raw K^T, T and P in the canonical
//     no-swizzle K-major layout (8-row x 16-byte core matrices);
//   * sixteen compute warps, one per (TMEM lane quarter, column quarter), do the
//     TMEM round trips and the elementwise work; a product warp issues every
//     product and commits each group to an mbarrier (Z alone first, then Y,
//     U, the state update, O); a loader warp brings each chunk's q, k, v
//     with tensor copies a chunk ahead into double buffers;
//   * the prep block of a chunk comes by one bulk copy, a chunk ahead.
//
// Tensor memory (512 columns, one CTA an SM): S 0-127; Z 128-191, later the
// head|tail of U diag(e^{G_C-G} ik) (128-159 | 160-191); Y 192-255; U
// 256-319, later O; the head|tail of S 320-383 | 384-447; those of E and
// later of U 448-479 | 480-511.  Every region is rewritten only after the
// products that read it have completed.
//
// Every mbarrier wait is bounded: one that runs out reports
// GDN_DEVERR_TIMEOUT, and the CTA stops without writing outputs or state,
// frees its tensor memory and returns.
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_chunk_common.cuh"
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_ptx.cuh"

namespace gdn {

namespace {

constexpr int TC_WARPS = 8;
constexpr int TC_THREADS = TC_WARPS * 32;
// the chunk kernel: sixteen compute warps, one a (TMEM lane quarter, column
// quarter), a warp that issues the tensor-core products and a warp that
// copies the next chunk's q, k and v into shared memory
constexpr int TCC_WARPS = 16;
constexpr int TCC_THREADS = TCC_WARPS * 32;
constexpr int TCW_THREADS = TCC_THREADS + 64;
constexpr uint32_t kTmemCols = 512;

// TMEM columns.  O accumulates into U's columns once U is split; E's and
// then U's heads and tails share 448-511 (S's split is read by the Z and Y
// products while E is formed, and written again while O's product still
// reads U's split); W's take Z's columns.
constexpr uint32_t C_S = 0, C_Z = 128, C_Y = 192, C_U = 256, C_SH = 320, C_SL = 384;
constexpr uint32_t C_EH = 448, C_EL = 480, C_UH = 448, C_UL = 480, C_WH = 128, C_WL = 160;

// Byte offset of element (row, k) in a canonical K-major tile with K columns.
template <int K> __device__ __forceinline__ int cm_off(int row, int k)
{
    return ((((row >> 3) * (K / 8)) + (k >> 3)) << 7) + ((row & 7) << 4) + ((k & 7) << 1);
}

// One chunk's state-free terms, as the prep kernel writes them to the
// workspace and as the chunk kernel takes them into shared memory with one
// bulk copy: P and T = (I + A)^{-1} split into bf16 heads and tails, in the
// canonical K-major layout the tensor cores read; the gates; the norm scales;
// a header naming the chunk (sequence, first token in it) the unit holds.
struct PW {
    static constexpr int PH = 0;                    // bf16 [64][64] P head, tail, T head, tail
    static constexpr int PL = PH + CK * CK * 2;
    static constexpr int TH = PL + CK * CK * 2;
    static constexpr int TL = TH + CK * CK * 2;
    static constexpr int GATES = TL + CK * CK * 2;  // fp32 [G | beta | e^G | e^{G_C - G}] x CK
    static constexpr int IQ = GATES + 4 * CK * 4;   // fp32 q norm scales (with 1/sqrt(dk)) [CK]
    static constexpr int IK = IQ + CK * 4;          // fp32 k norm scales [CK]
    static constexpr int HDR = IK + CK * 4;         // int32 sequence, first token of the chunk in it
    static constexpr int BYTES = (HDR + 8 + 127) & ~127;
};
static_assert(PW::BYTES % 128 == 0, "prep blocks stay 128-byte aligned");

// Workspace units of one value head: sequence s's chunk j is unit
// cu_seqlens[s] / CK + s + j.  Distinct for every chunk of nondecreasing
// cu_seqlens; ceil(total_tokens / CK) + nseq units cover every index.
__host__ __device__ __forceinline__ long long prep_units(int nseq, int total_tokens)
{
    return (long long)(total_tokens + CK - 1) / CK + nseq;
}
__device__ __forceinline__ int unit_base(const int32_t *cu, int s) { return cu[s] / CK + s; }

// Shared-memory layout of the chunk kernel, byte offsets.
struct TS {
    // raw K then raw Q of a chunk, each as two 64-token x 64-dk halves of
    // 128-byte rows in the 128-byte-swizzled K-major layout (what a tensor
    // copy with that swizzle writes, 1024-byte aligned)
    static constexpr int HALF = CK * 64 * 2;      // 8 KiB
    static constexpr int KQ_BYTES = 4 * HALF;     // K dk 0-63 | K dk 64-127 | Q dk 0-63 | Q dk 64-127
    static constexpr int KQ = 0;                  // two of them, chunk parity
    static constexpr int KT_BYTES = CD * CK * 2;  // bf16 [128 = dk][64 = tokens]: raw K transposed
    static constexpr int KT = KQ + 2 * KQ_BYTES;  // two of them, chunk parity
    static constexpr int PB = KT + 2 * KT_BYTES;  // two prep blocks (PW), chunk parity
    static constexpr int BARS = PB + 2 * PW::BYTES; // mbarriers: Z, U, O, prep block 0, 1, S;
                                                    // S's split, E, U's split ready; inputs 0, 1;
                                                    // output tile free
    static constexpr int TADDR = BARS + 96;       // the TMEM base address
    static constexpr int BYTES = TADDR + 16;
    static constexpr int STAGE = (BYTES + 127) & ~127; // raw v, [CK][CD], two of them, chunk parity
    static constexpr int OUTS = STAGE + 2 * CK * CD * 2; // bf16 outputs of a chunk, [CK][CD]
    static constexpr int USED = OUTS + CK * CD * 2;
    static constexpr int TOTAL = USED + 1024;     // the base rounded up to 1024 bytes
};
static_assert(TS::TOTAL <= 227 * 1024, "shared memory");
static_assert(TS::KQ % 1024 == 0 && TS::KQ_BYTES % 1024 == 0 && TS::HALF % 1024 == 0, "swizzled tiles");
static_assert(TS::STAGE % 128 == 0 && TS::OUTS % 16 == 0, "copy destinations");
static_assert(TS::BARS % 8 == 0 && TS::KT % 1024 == 0 && TS::PB % 128 == 0, "alignment");

// Shared-memory layout of the prep kernel, byte offsets.
struct PS {
    static constexpr int LDQ = CD + 8;            // row stride (bf16) of q and k: rows 272 B apart, so
                                                  // a fragment's 8 rows fall in distinct banks
    static constexpr int RQ = 0;                  // bf16 [CK][LDQ] raw q, k (row-major)
    static constexpr int RK = RQ + CK * LDQ * 2;
    // once [K|Q] K^T is in registers, q and k are dead: A and the decay / T take their place
    static constexpr int AF = 0;                  // fp32 A [t][s] (upper blocks: scratch)
    static constexpr int XF = AF + CK * LDF * 4;  // fp32 decay, then T [t][s]
    static constexpr int QK_END = RK + CK * LDQ * 2;
    static constexpr int AX_END = XF + CK * LDF * 4;
    static constexpr int GATES = QK_END > AX_END ? QK_END : AX_END;
    static constexpr int IQ = GATES + 4 * CK * 4;
    static constexpr int IK = IQ + CK * 4;
    static constexpr int TOTAL = IK + CK * 4;
};

// ---- tcgen05 wrappers ----
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t sbo)
{
    // start >> 4 | leading offset (K-adjacent core matrices: 128 B) >> 4 | stride offset >> 4 | version 1
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
// the same for a K-major operand in the 128-byte-swizzled layout: 8-row
// groups 1024 bytes apart (stride offset); the leading offset is unused
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFF) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
// one box of a 3-D tensor map into shared memory, counted on `bar`
__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3, %4}], [%5];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
                 : "memory");
}
// The tensor maps of a call: q and k [tokens][hk][dk], boxes of 64 dk x 1
// head x 64 tokens, 128-byte swizzle; v [tokens][hv][dv], 128 x 1 x 64.
struct ChunkMaps {
    CUtensorMap q, k, v;
};
// D fp32, A and B bf16, both K-major, M = 128, N = n
__host__ __device__ constexpr uint32_t idesc_bf16(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
// A from tensor memory, B from shared memory
__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)acc)
                 : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// shared-memory writes made visible to the tensor cores' reads
__device__ __forceinline__ void smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive columns of this thread's lane
__device__ __forceinline__ void tld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
                   "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
                   "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}
// 16 consecutive columns of this thread's lane
__device__ __forceinline__ void tld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                 "[%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tst8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tst32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                 "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
                 "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
                 "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
__device__ __forceinline__ void tst16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                 "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}
__device__ __forceinline__ void tst_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 fp32 values -> their bf16 head and tail as 16 + 16 packed pairs
__device__ __forceinline__ void split32(const float (&v)[32], uint32_t (&hi)[16], uint32_t (&lo)[16])
{
#pragma unroll
    for (int j = 0; j < 16; ++j)
        split2(v[2 * j], v[2 * j + 1], hi[j], lo[j]);
}

// ---------------------------------------------------------------------------
// The prep kernel: one CTA per (workspace unit, value head).  It finds the
// chunk its unit holds, then forms the chunk's state-free terms: the gates,
// the norm scales, [K|Q] K^T on the tensor cores (mma.sync; exact bf16
// products, fp32 sums), A and P from it, T = (I + A)^{-1} by the blocked
// inverse, and writes them with a header to the unit.  Units that hold no
// chunk get a header that names none.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(TC_THREADS, 5) gdn_chunk_prep_kernel(const PrefillArgs p, unsigned char *work,
                                                                    int units)
{
    extern __shared__ __align__(128) unsigned char smem[];
    bf16 *const RQ = reinterpret_cast<bf16 *>(smem + PS::RQ);
    bf16 *const RK = reinterpret_cast<bf16 *>(smem + PS::RK);
    float *const AF = reinterpret_cast<float *>(smem + PS::AF);
    float *const XF = reinterpret_cast<float *>(smem + PS::XF);
    float *const GATES = reinterpret_cast<float *>(smem + PS::GATES);
    float *const IQ = reinterpret_cast<float *>(smem + PS::IQ);
    float *const IK = reinterpret_cast<float *>(smem + PS::IK);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
    const int u = blockIdx.x / p.hv, h = blockIdx.x - (blockIdx.x / p.hv) * p.hv;
    unsigned char *const blk = work + ((size_t)h * units + u) * PW::BYTES;
    int32_t *const hdr = reinterpret_cast<int32_t *>(blk + PW::HDR);
    wait_prior_grid();
    // The chunk kernel may launch now (every earlier kernel is complete): its
    // CTAs set up and load their state beside this grid's last CTAs, and wait
    // for this grid to complete before they read a unit.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // the sequence whose units start at or before u: the last s with base(s) <= u
    int lo = 0, hi = p.nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (unit_base(p.cu_seqlens, mid) <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int s = lo;
    const int t0 = p.cu_seqlens[s], t1 = p.cu_seqlens[s + 1];
    const int j = u - unit_base(p.cu_seqlens, s);
    const int c0 = CK * j;
    if (t0 < 0 || t1 < t0 || t1 > p.total_tokens || j < 0 || c0 >= t1 - t0) {
        if (tid == 0)
            hdr[0] = -1, hdr[1] = -1;
        return;
    }
    const int n = min(CK, t1 - t0 - c0);
    const int hq = h / (p.hv / p.hk);
    const bf16 *const qg = reinterpret_cast<const bf16 *>(p.q);
    const bf16 *const kg = reinterpret_cast<const bf16 *>(p.k);

    // the chunk's raw q and k rows (zeros past its tokens), 16 bytes a copy
    for (int e = tid; e < 2 * CK * (CD / 8); e += TC_THREADS) {
        const int which = e / (CK * (CD / 8)), rem = e - which * (CK * (CD / 8));
        const int tt = rem / (CD / 8), jj = rem - tt * (CD / 8);
        const bool live = tt < n;
        const size_t tok = (size_t)(t0 + c0 + (live ? tt : 0));
        const bf16 *src = (which == 0 ? qg : kg) + (tok * p.hk + hq) * CD;
        bf16 *dst = (which == 0 ? RQ : RK) + tt * PS::LDQ;
        cp_async16(dst + 8 * jj, src + 8 * jj, live ? 16 : 0);
    }
    cp_async_commit();
    if (warp == 0) {
        // the gates
        const bf16 *const ag = reinterpret_cast<const bf16 *>(p.a);
        const bf16 *const bg = reinterpret_cast<const bf16 *>(p.b);
        bf16 ra[2], rb[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int tt = lane + 32 * i;
            ra[i] = rb[i] = from_f<bf16>(0.f);
            if (tt < n) {
                const size_t idx = (size_t)(t0 + c0 + tt) * p.hv + h;
                ra[i] = ag[idx], rb[i] = bg[idx];
            }
        }
        chunk_gates(GATES, ra, rb, n, expf(p.A_log[h]), p.dt_bias[h], lane);
    }
    cp_async_wait_all();
    __syncthreads();

    // norm scales, four tokens a warp at a time: lanes 8j .. 8j + 7 take
    // token j's dk 8p .. 8p + 7 and 64 + 8p .. 64 + 8p + 7 (p = lane & 7),
    // 16 bytes a load, and sum over the eight
    {
        const float qscale = 1.0f / sqrtf((float)CD);
        const int p8 = lane & 7;
#pragma unroll
        for (int i = 0; i < CK / (4 * TC_WARPS); ++i) {
            const int tt = 4 * (TC_WARPS * i + warp) + (lane >> 3);
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                const uint4 qv = *reinterpret_cast<const uint4 *>(RQ + tt * PS::LDQ + 64 * hlf + 8 * p8);
                const uint4 kv = *reinterpret_cast<const uint4 *>(RK + tt * PS::LDQ + 64 * hlf + 8 * p8);
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // a bf16 pair to fp32 exactly: the low half shifted up, the high half masked
                    const float q0 = __uint_as_float(qw[e] << 16), q1 = __uint_as_float(qw[e] & 0xffff0000u);
                    const float k0 = __uint_as_float(kw[e] << 16), k1 = __uint_as_float(kw[e] & 0xffff0000u);
                    sq = fmaf(q1, q1, fmaf(q0, q0, sq));
                    sk = fmaf(k1, k1, fmaf(k0, k0, sk));
                }
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (p8 == 0)
                IQ[tt] = qscale * rsqrtf(sq + kEps), IK[tt] = rsqrtf(sk + kEps);
        }
    }
    // [K|Q] K^T over the tiles at or below the diagonal only: row block R
    // (rows 16R .. 16R + 15) has the 16 x 8 tiles nt = 0 .. 2R + 1 there, 20
    // of K's 32 and 20 of Q's.  Warp role r = warp & 3 (K's rows for warps
    // 0-3, Q's for 4-7) takes five: two of block bA from column tile nA and
    // three of block bB from nB,
    //   r 0: block 0 tiles 0-1, block 3 tiles 0-2;  r 1: block 1 tiles 0-1, block 3 tiles 3-5;
    //   r 2: block 1 tiles 2-3, block 2 tiles 0-2;  r 3: block 3 tiles 6-7, block 2 tiles 3-5.
    const bool isq = warp >= 4;
    const bf16 *const X = isq ? RQ : RK;
    const int r = warp & 3;
    const int bA = r == 0 ? 0 : r == 3 ? 3 : 1, nA = r == 2 ? 2 : r == 3 ? 6 : 0;
    const int bB = r < 2 ? 3 : 2, nB = (r & 1) ? 3 : 0;
    float d[5][4];
#pragma unroll
    for (int i = 0; i < 5; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            d[i][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < CD / 16; ++ks) {
        uint32_t aa[4], ab[4];
        lda(aa, X, PS::LDQ, 16 * bA, 16 * ks, g, c);
        lda(ab, X, PS::LDQ, 16 * bB, 16 * ks, g, c);
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            uint32_t b0, b1;
            ldb(b0, b1, RK, PS::LDQ, 8 * (i < 2 ? nA + i : nB + i - 2), 16 * ks, g, c);
            if (i < 2)
                mma16816(d[i], aa[0], aa[1], aa[2], aa[3], b0, b1);
            else
                mma16816(d[i], ab[0], ab[1], ab[2], ab[3], b0, b1);
        }
    }
    __syncthreads(); // every warp's products are in registers: q and k are dead

    // A[t][s] = beta_t e^{G_t-G_s} ik_t ik_s (k_t . k_s), s < t, into AF (over
    // q and k); P[t][s] = e^{G_t-G_s} iq_t ik_s (q_t . k_s), s <= t, split, to
    // the unit; the decay formed where it is used.  A row's gate and scale,
    // and a column pair's, are loaded once (the stores into AF may alias them
    // for the compiler).  A's tiles above the diagonal are never read; P's
    // are zero, written below.
    const float *const BE = GATES + CK;
    float gt[2][2], sc[2][2]; // [block A or B][row g or g + 8]
#pragma unroll
    for (int w = 0; w < 2; ++w)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int t = 16 * (w == 0 ? bA : bB) + g + 8 * hh;
            gt[w][hh] = GATES[t];
            sc[w][hh] = isq ? IQ[t] : IK[t] * BE[t];
        }
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        const int w = i < 2 ? 0 : 1;
        const int m0 = 16 * (w == 0 ? bA : bB);
        const int s0 = 8 * (i < 2 ? nA + i : nB + i - 2) + 2 * c;
        const float2 gs = *reinterpret_cast<const float2 *>(GATES + s0);
        const float2 ks = *reinterpret_cast<const float2 *>(IK + s0);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int t = m0 + g + 8 * hh;
            const float nt_ = sc[w][hh];
            const bool in0 = isq ? s0 <= t : s0 < t, in1 = isq ? s0 + 1 <= t : s0 + 1 < t;
            const float x = in0 ? expf(gt[w][hh] - gs.x) * nt_ * ks.x * d[i][2 * hh] : 0.f;
            const float y = in1 ? expf(gt[w][hh] - gs.y) * nt_ * ks.y * d[i][2 * hh + 1] : 0.f;
            if (!isq) {
                *reinterpret_cast<float2 *>(AF + t * LDF + s0) = make_float2(x, y);
            } else {
                uint32_t ph, pl;
                split2(x, y, ph, pl);
                *reinterpret_cast<uint32_t *>(blk + PW::PH + cm_off<CK>(t, s0)) = ph;
                *reinterpret_cast<uint32_t *>(blk + PW::PL + cm_off<CK>(t, s0)) = pl;
            }
        }
    }
    if (isq) {
        // P's 12 tiles wholly above the diagonal, three a Q warp: in order
        // block 0 tiles 2-7, block 1 tiles 4-7, block 2 tiles 6-7
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int k = 3 * r + j;
            const int R = k < 6 ? 0 : k < 10 ? 1 : 2, nt = k < 6 ? k + 2 : k < 10 ? k - 2 : k - 4;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = 16 * R + g + 8 * hh, s0 = 8 * nt + 2 * c;
                *reinterpret_cast<uint32_t *>(blk + PW::PH + cm_off<CK>(t, s0)) = 0u;
                *reinterpret_cast<uint32_t *>(blk + PW::PL + cm_off<CK>(t, s0)) = 0u;
            }
        }
    }
    __syncthreads();
    if (tid < CK) {
        t_diagonal(AF, XF, tid);
    } else {
        // meanwhile the gates and norm scales go to the unit
        float *const og = reinterpret_cast<float *>(blk + PW::GATES);
        for (int e = tid - CK; e < 4 * CK; e += TC_THREADS - CK)
            og[e] = GATES[e];
        if (tid >= TC_THREADS - CK) {
            const int t = tid - (TC_THREADS - CK);
            reinterpret_cast<float *>(blk + PW::IQ)[t] = IQ[t];
            reinterpret_cast<float *>(blk + PW::IK)[t] = IK[t];
        }
    }
    __syncthreads();
    t_below_diagonal(AF, XF, warp, g, c);
    // T's lower triangle, split, to the unit, one 16-byte row of a core
    // matrix a thread: a warp writes four adjacent core matrices (512
    // contiguous bytes); piece p = row group 8 rg, core columns 4 (q & 1) ..
    // + 3 with q = p / 32, lane: row lane & 7, core column (lane >> 3)
#pragma unroll
    for (int i = 0; i < CK * CK / 8 / TC_THREADS; ++i) {
        const int pc = tid + TC_THREADS * i, q = pc >> 5;
        const int t = 8 * (q >> 1) + (lane & 7), k8 = 4 * (q & 1) + (lane >> 3);
        uint4 th = make_uint4(0u, 0u, 0u, 0u), tl = th;
        if (8 * k8 <= t) {
            const float4 v0 = *reinterpret_cast<const float4 *>(XF + t * LDF + 8 * k8);
            const float4 v1 = *reinterpret_cast<const float4 *>(XF + t * LDF + 8 * k8 + 4);
            const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint32_t h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                split2(8 * k8 + 2 * e <= t ? v[2 * e] : 0.f, 8 * k8 + 2 * e + 1 <= t ? v[2 * e + 1] : 0.f, h[e],
                       l[e]);
            th = make_uint4(h[0], h[1], h[2], h[3]);
            tl = make_uint4(l[0], l[1], l[2], l[3]);
        }
        *reinterpret_cast<uint4 *>(blk + PW::TH + cm_off<CK>(t, 8 * k8)) = th;
        *reinterpret_cast<uint4 *>(blk + PW::TL + cm_off<CK>(t, 8 * k8)) = tl;
    }
    if (tid == 0)
        hdr[0] = s, hdr[1] = c0;
}

// the sixteen compute warps (TCC_THREADS = 512 threads) meet at named
// barrier 1; the _or form also returns whether any of them passed true
static_assert(TCC_THREADS == 512, "the named barriers below count 512 threads");
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
__device__ __forceinline__ bool compute_sync_or(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 512, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v)
                 : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(TCW_THREADS, 1) gdn_chunked_tc_kernel(const PrefillArgs p,
                                                                      const unsigned char *work, int units,
                                                                      const __grid_constant__ ChunkMaps maps)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *const smem = smem_raw + ((1024u - (sm_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char *const KQ = smem + TS::KQ;
    unsigned char *const KT = smem + TS::KT;
    uint64_t *const bars = reinterpret_cast<uint64_t *>(smem + TS::BARS);
    uint32_t *const taddr_slot = reinterpret_cast<uint32_t *>(smem + TS::TADDR);
    bf16 *const RV = reinterpret_cast<bf16 *>(smem + TS::STAGE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, cq = warp >> 2; // compute warps: TMEM lane quarter, column quarter
    const int row = 32 * quarter + lane; // this thread's state row (its TMEM lane)
    const int seq = blockIdx.x / p.hv, h = blockIdx.x - seq * p.hv;
    const int hq = h / (p.hv / p.hk);
    // Everything up to the first chunk's prep block reads only this call's
    // inputs, which the prep kernel does not write: it runs before
    // wait_prior_grid, beside the prep kernel's last CTAs (which let this grid
    // launch only after their own wait, so every earlier kernel is complete).

    const int t0 = p.cu_seqlens[seq], t1 = p.cu_seqlens[seq + 1];
    const bool range_ok = t0 >= 0 && t1 >= t0 && t1 <= p.total_tokens;
    const int rs = p.read_slot[seq];
    const bool in_place = p.write_slot == nullptr;
    const int ws = in_place ? rs : p.write_slot[seq];
    const int cls = range_ok ? classify_row(rs, ws, p.num_slots, in_place) : -1;
    bf16 *const out = reinterpret_cast<bf16 *>(p.out);
    const size_t out_tok = (size_t)p.hv * CD;
    if (cls != 1) {
        // padding or bad: zero outputs (when the token range is sane), no slot touched
        if (cls < 0 && h == 0 && tid == 0)
            report(p.err, GDN_DEVERR_BAD_SLOT);
        if (range_ok) {
            const long long n_out = (long long)(t1 - t0) * CD;
            for (long long e = tid; e < n_out; e += TCW_THREADS)
                out[(size_t)(t0 + e / CD) * out_tok + (size_t)h * CD + (size_t)(e % CD)] = from_f<bf16>(0.f);
        }
        return;
    }

    const int L = t1 - t0;
    const unsigned char *const hwork = work + (size_t)h * units * PW::BYTES;
    const int ubase = unit_base(p.cu_seqlens, seq);

    // tensor memory (all 512 columns) and the products' mbarriers
    const uint32_t bar_z = sm_addr(&bars[0]), bar_u = sm_addr(&bars[1]), bar_o = sm_addr(&bars[2]);
    const uint32_t bar_pb[2] = {sm_addr(&bars[3]), sm_addr(&bars[4])};
    const uint32_t bar_s = sm_addr(&bars[5]);
    // compute warps -> product warp: S's split, E's split, U's and W's splits are in TMEM
    const uint32_t bar_sready = sm_addr(&bars[6]), bar_eready = sm_addr(&bars[7]);
    const uint32_t bar_wready = sm_addr(&bars[8]);
    // loader warp -> compute warps: a chunk's q, k and v are in shared memory (chunk parity)
    const uint32_t bar_in[2] = {sm_addr(&bars[9]), sm_addr(&bars[10])};
    // loader warp -> compute warps: it has stored the output tile (one completion a chunk but the last)
    const uint32_t bar_osfree = sm_addr(&bars[11]);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sm_addr(taddr_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        mbar_init(bar_z, 1);
        mbar_init(bar_u, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_sready, TCC_WARPS);
        mbar_init(bar_eready, TCC_WARPS);
        mbar_init(bar_wready, TCC_WARPS);
        mbar_init(bar_in[0], 1);
        mbar_init(bar_in[1], 1);
        mbar_init(bar_osfree, 1);
        mbar_init(bar_pb[0], 1);
        mbar_init(bar_pb[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tbase = *taddr_slot;
    const uint32_t tlane = tbase + ((uint32_t)(32 * quarter) << 16); // this warp's 32 lanes

    // the state in: row `row`, columns 32*cq .. 32*cq + 31 (compute warps)
    const size_t slot_floats = (size_t)p.hv * CD * CD;
    const size_t head_off = (size_t)h * CD * CD;
    if (warp < TCC_WARPS) {
        const float *S0 = p.pool + (size_t)rs * slot_floats + head_off + (size_t)row * CD + 32 * cq;
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = *reinterpret_cast<const float4 *>(S0 + 4 * i);
            r[4 * i] = __float_as_uint(v.x), r[4 * i + 1] = __float_as_uint(v.y);
            r[4 * i + 2] = __float_as_uint(v.z), r[4 * i + 3] = __float_as_uint(v.w);
        }
        tst32(tlane + C_S + 32 * cq, r);
        tst_wait();
    }

    // The raw q, k, v of the chunk starting at token cn into the buffers of
    // parity `buf`, by five tensor copies counted on bar_in[buf] (one
    // thread): k and q as two 128-byte-swizzled dk halves each, v row-major.
    // A box reads past the sequence into the next one's tokens (zeros past the
    // last token): those rows are neutralised where they are used (E is zero
    // and K^T has zeros for tokens past the chunk's end).
    auto load_chunk = [&](int cn, int buf) {
        const uint32_t bar = bar_in[buf];
        const uint32_t kq = sm_addr(KQ + buf * TS::KQ_BYTES);
        mbar_arrive_tx(bar, (uint32_t)(TS::KQ_BYTES + CK * CD * 2));
        const int tok = t0 + cn;
        tma_load3(kq, &maps.k, 0, hq, tok, bar);
        tma_load3(kq + TS::HALF, &maps.k, 64, hq, tok, bar);
        tma_load3(kq + 2 * TS::HALF, &maps.q, 0, hq, tok, bar);
        tma_load3(kq + 3 * TS::HALF, &maps.q, 64, hq, tok, bar);
        tma_load3(sm_addr(RV + buf * CK * CD), &maps.v, 0, h, tok, bar);
    };
    // K^T of the chunk (nn tokens) whose K rows are in K | Q tile `buf`, into
    // K^T buffer `buf`: a warp transposes four 8x8 blocks a step (ldmatrix
    // .trans from the swizzled rows: lane l gets tokens 2 (l % 4) and
    // 2 (l % 4) + 1 of dk row l / 4), zeroes tokens past nn, and stores each
    // block as one word of a canonical core-matrix row
    auto build_kt = [&](int buf, int nn) {
        unsigned char *const kt = KT + buf * TS::KT_BYTES;
        const unsigned char *const kq = KQ + buf * TS::KQ_BYTES;
        for (int g = warp; g < (CK / 8) * (CD / 8) / 4; g += TCC_WARPS) {
            const int m = 4 * g + (lane >> 3);
            const int r = 8 * (m / (CD / 8)) + (lane & 7), jb = m % (CD / 8); // token row, 16-byte piece
            const uint32_t src = sm_addr(kq + (jb >> 3) * TS::HALF + r * 128 + (((jb & 7) ^ (r & 7)) << 4));
            uint32_t w[4];
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(src)
                         : "memory");
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int mi = 4 * g + i, tb = mi / (CD / 8), jbi = mi % (CD / 8);
                const int s0 = 8 * tb + 2 * (lane & 3); // tokens s0, s0 + 1
                uint32_t v = w[i];
                if (s0 >= nn)
                    v = 0;
                else if (s0 + 1 >= nn)
                    v &= 0xFFFFu;
                *reinterpret_cast<uint32_t *>(kt + cm_off<CK>(8 * jbi + (lane >> 2), s0)) = v;
            }
        }
    };
    // the prep block of chunk cj into the shared prep block of its parity (one
    // bulk copy; its previous chunk's products, which read it, are done)
    auto prep_copy = [&](int cj) {
        if (tid == 0) {
            smem_to_async();
            const uint32_t bar = bar_pb[cj & 1];
            mbar_arrive_tx(bar, (uint32_t)PW::BYTES);
            bulk_load(sm_addr(smem + TS::PB + (cj & 1) * PW::BYTES), hwork + (size_t)(ubase + cj) * PW::BYTES,
                      (uint32_t)PW::BYTES, bar);
        }
    };
    // The outputs of a chunk leave in two steps: each compute thread puts
    // its row `row` of O (in U's columns), tokens 16*cq .. 16*cq + 15, into
    // the shared output tile (put_outputs); then threads store 16-byte pieces
    // of the tile's token rows (store_outputs).
    bf16 *const OS = reinterpret_cast<bf16 *>(smem + TS::OUTS);
    auto put_outputs = [&]() {
        float o[16];
        tld16(tlane + C_U + 16 * cq, o);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            OS[(16 * cq + i) * CD + row] = from_f<bf16>(o[i]);
    };
    // (16-byte stores when `out` is 16-byte aligned, as its rows then are;
    // the call does not require it, so 2-byte stores otherwise)
    const bool out16 = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    auto store_outputs = [&](int cbase, int nn, int me, int nthr) {
        if (out16) {
            for (int e = me; e < nn * (CD / 8); e += nthr) {
                const int t = e / (CD / 8), j = e % (CD / 8);
                *reinterpret_cast<uint4 *>(out + (size_t)(t0 + cbase + t) * out_tok + (size_t)h * CD + 8 * j) =
                    *reinterpret_cast<const uint4 *>(OS + t * CD + 8 * j);
            }
        } else {
            for (int e = me; e < nn * CD; e += nthr)
                out[(size_t)(t0 + cbase + e / CD) * out_tok + (size_t)h * CD + (e % CD)] = OS[e];
        }
    };
    if (L > 0 && warp == TCC_WARPS + 1 && lane == 0)
        load_chunk(0, 0); // q, k and v are this call's inputs: no earlier kernel writes them
    wait_prior_grid(); // the prep kernel's units are complete

    // the prep kernel's units of this sequence must name its chunks (they do
    // unless cu_seqlens decreases somewhere): otherwise it counts as bad
    bool named = true;
    for (int j = tid; CK * j < L; j += TCW_THREADS) {
        const int32_t *hd = reinterpret_cast<const int32_t *>(hwork + (size_t)(ubase + j) * PW::BYTES + PW::HDR);
        named = named && ubase + j < units && hd[0] == seq && hd[1] == CK * j;
    }
    if (!__syncthreads_and(named)) {
        if (L > 0 && warp == TCC_WARPS + 1 && lane == 0)
            mbar_wait(bar_in[0], 0u); // the first chunk's copies land before the CTA ends
        if (h == 0 && tid == 0)
            report(p.err, GDN_DEVERR_BAD_SLOT);
        for (long long e = tid; e < (long long)L * CD; e += TCW_THREADS)
            out[(size_t)(t0 + e / CD) * out_tok + (size_t)h * CD + (size_t)(e % CD)] = from_f<bf16>(0.f);
        cp_async_wait_all();
        tc_before_sync();
        __syncthreads();
        if (warp == 0)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols) : "memory");
        return;
    }
    bool in_late = false; // a wait for the loader's copies ran out
    if (L > 0) {
        prep_copy(0);
        // chunk c's inputs complete phase c / 2 of bar_in[c % 2]
        if (warp < TCC_WARPS) {
            in_late = !__all_sync(0xffffffffu, mbar_wait(bar_in[0], 0u));
            if (!in_late)
                build_kt(0, min(CK, L));
        }
    }

    // this chunk's prep block, by chunk parity
    auto pblock = [&](int ci) { return smem + TS::PB + (ci & 1) * PW::BYTES; };

    if (warp < TCC_WARPS) {
        // ======================= compute warps =======================
        bool abort = false;
        int n_prev = 0;
#pragma unroll 1
        for (int c0 = 0; c0 < L; c0 += CK) {
            const int ci = c0 / CK;
            const int n = min(CK, L - c0);
            unsigned char *const PBc = pblock(ci);
            const float *const GG = reinterpret_cast<const float *>(PBc + PW::GATES); // this chunk's gates
            const float *const IQ = reinterpret_cast<const float *>(PBc + PW::IQ);
            const float *const IK = reinterpret_cast<const float *>(PBc + PW::IK);
            const float *const BE = GG + CK;
            const float *const EG = GG + 2 * CK;
            const float *const EC = GG + 3 * CK;
            const bool more = c0 + CK < L;

            // ---- (0) the previous chunk's state update is done: S's head
            // and tail for the product warp (this chunk's K | Q and K^T are
            // in place) ----
            bool late = in_late || (ci > 0 && !mbar_wait(bar_s, (uint32_t)((ci - 1) & 1)));
            if (late)
                report(p.err, GDN_DEVERR_TIMEOUT);
            if (compute_sync_or(late)) {
                abort = true;
                break;
            }
            tc_after_sync();
            {
                float sv[32];
                uint32_t hi[16], lo[16];
                tld32(tlane + C_S + 32 * cq, sv);
                split32(sv, hi, lo);
                tst16(tlane + C_SH + 16 * cq, hi);
                tst16(tlane + C_SL + 16 * cq, lo);
            }
            tst_wait();
            smem_to_async(); // K^T, written through the generic proxy
            tc_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_sready);

            // ---- (2) the previous chunk's outputs, while Z runs; this
            // chunk's prep block; then E from Z, one state row a thread ----
            // the previous chunk's O is done, and the loader warp has stored
            // the output tile of the chunk before it
            late = __any_sync(0xffffffffu, (ci > 0 && !mbar_wait(bar_o, (uint32_t)((ci - 1) & 1))) ||
                                               (ci > 1 && !mbar_wait(bar_osfree, (uint32_t)((ci - 2) & 1))));
            if (ci > 0 && !late)
                put_outputs(); // warp-wide TMEM loads: the warp agrees on `late`
            late = late || !mbar_wait(bar_pb[ci & 1], (uint32_t)((ci >> 1) & 1)) ||
                   !mbar_wait(bar_z, (uint32_t)(ci & 1));
            if (late)
                report(p.err, GDN_DEVERR_TIMEOUT);
            if (compute_sync_or(late)) {
                abort = true;
                break;
            }
            tc_after_sync();
            if (more)
                prep_copy(ci + 1); // its block's last readers, the previous chunk's products, are done
            {
                const bf16 *const rv = RV + (ci & 1) * CK * CD;
                float z[16];
                tld16(tlane + C_Z + 16 * cq, z);
                uint32_t eh[8], el[8];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const int t = 16 * cq + i; // even: the pairs below are 8-byte loads
                    const float v0 = __bfloat162float(rv[t * CD + row]), v1 = __bfloat162float(rv[(t + 1) * CD + row]);
                    const float2 be = *reinterpret_cast<const float2 *>(BE + t);
                    const float2 eg = *reinterpret_cast<const float2 *>(EG + t);
                    const float2 ik = *reinterpret_cast<const float2 *>(IK + t);
                    // tokens past the chunk's end: E is zero (their v and Z may
                    // be the next sequence's)
                    const float e0 = t < n ? be.x * (v0 - eg.x * ik.x * z[i]) : 0.f;
                    const float e1 = t + 1 < n ? be.y * (v1 - eg.y * ik.y * z[i + 1]) : 0.f;
                    split2(e0, e1, eh[i / 2], el[i / 2]);
                }
                tst8(tlane + C_EH + 8 * cq, eh);
                tst8(tlane + C_EL + 8 * cq, el);
                tst_wait();
            }
            smem_to_async(); // v read here, before the loader's next copy into its buffer
            tc_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_eready);
            {
                // S scaled by e^{G_C} while U's product runs: no product reads
                // or writes S's own columns between its split above and the
                // state update, which waits for wready (after the wait below)
                const float gC = EG[CK - 1];
                float sv[32];
                uint32_t r[32];
                tld32(tlane + C_S + 32 * cq, sv);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r[i] = __float_as_uint(sv[i] * gC);
                tst32(tlane + C_S + 32 * cq, r);
            }

            // ---- (3) U's head and tail (for O), those of U diag(e^{G_C-G}
            // ik) (for S), Y diag(e^G iq) into U's columns (where O
            // accumulates) ----
            late = !mbar_wait(bar_u, (uint32_t)(ci & 1)); // Y's products came before U's
            if (late)
                report(p.err, GDN_DEVERR_TIMEOUT);
            if (compute_sync_or(late)) {
                abort = true;
                break;
            }
            tc_after_sync();
            {
                float u[16];
                tld16(tlane + C_U + 16 * cq, u);
                uint32_t uh[8], ul[8], wh[8], wl[8];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const int t = 16 * cq + i;
                    const float2 ec = *reinterpret_cast<const float2 *>(EC + t);
                    const float2 ik = *reinterpret_cast<const float2 *>(IK + t);
                    split2(u[i], u[i + 1], uh[i / 2], ul[i / 2]);
                    split2(u[i] * ec.x * ik.x, u[i + 1] * ec.y * ik.y, wh[i / 2], wl[i / 2]);
                }
                tst8(tlane + C_UH + 8 * cq, uh);
                tst8(tlane + C_UL + 8 * cq, ul);
                tst8(tlane + C_WH + 8 * cq, wh);
                tst8(tlane + C_WL + 8 * cq, wl);
                {
                    float y[16];
                    uint32_t yo[16];
                    tld16(tlane + C_Y + 16 * cq, y);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const int t = 16 * cq + i;
                        const float2 eg = *reinterpret_cast<const float2 *>(EG + t);
                        const float2 iq = *reinterpret_cast<const float2 *>(IQ + t);
                        yo[i] = __float_as_uint(y[i] * eg.x * iq.x);
                        yo[i + 1] = __float_as_uint(y[i + 1] * eg.y * iq.y);
                    }
                    tst16(tlane + C_U + 16 * cq, yo);
                }
                tst_wait(); // and S's scaled rows, stored during the U product

            }
            tc_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_wready);
            n_prev = n;
            if (more) {
                // the next chunk's K^T, beside the products (they read the
                // other K^T buffer), once the loader warp has its rows in
                // (a failed wait leaves it unbuilt and ends the loop at the
                // next chunk's top; the warp agrees, its loads are warp-wide)
                in_late = !__all_sync(0xffffffffu, mbar_wait(bar_in[(ci + 1) & 1], (uint32_t)(((ci + 1) >> 1) & 1)));
                if (!in_late)
                    build_kt((ci + 1) & 1, min(CK, L - c0 - CK));
            }
        }

        if (!abort && L > 0) {
            const int last = (L - 1) / CK;
            const bool late = !mbar_wait(bar_o, (uint32_t)(last & 1)); // after S's product
            if (late)
                report(p.err, GDN_DEVERR_TIMEOUT);
            abort = compute_sync_or(late);
            if (!abort) {
                tc_after_sync();
                // the loader warp's store of the tile before (none with one chunk)
                const bool tile_late =
                    __any_sync(0xffffffffu, last > 0 && !mbar_wait(bar_osfree, (uint32_t)((last - 1) & 1)));
                if (tile_late)
                    report(p.err, GDN_DEVERR_TIMEOUT);
                if (!tile_late)
                    put_outputs();
                compute_sync();
                if (!tile_late)
                    store_outputs(last * CK, n_prev, tid, TCC_THREADS);
            }
        }
        if (!abort) {
            // the final state, to the write slot (the read slot in place)
            float *Sd = p.pool + (size_t)ws * slot_floats + head_off + (size_t)row * CD + 32 * cq;
            float sv[32];
            tld32(tlane + C_S + 32 * cq, sv);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float4 *>(Sd + 4 * i) =
                    make_float4(sv[4 * i], sv[4 * i + 1], sv[4 * i + 2], sv[4 * i + 3]);
        }
    } else if (warp == TCC_WARPS) {
        // ======================= product warp ========================
        // Per chunk: Z = S K^T (committed alone, E needs it first), Y = S
        // Q^T; U = E T^T (its commit covers Y's products too); S += W K,
        // then O += U P^T.  Each group waits for the compute warps' inputs.
#pragma unroll 1
        for (int c0 = 0; lane == 0 && c0 < L; c0 += CK) {
            const int ci = c0 / CK;
            unsigned char *const PBc = pblock(ci);
            if (!mbar_wait(bar_sready, (uint32_t)(ci & 1))) {
                report(p.err, GDN_DEVERR_TIMEOUT);
                break;
            }
            tc_after_sync();
            // K's and Q's swizzled halves: 16 dk (32 bytes) a step inside a half
            const uint32_t kq = sm_addr(KQ + (ci & 1) * TS::KQ_BYTES);
#pragma unroll
            for (int ks = 0; ks < CD / 16; ++ks) {
                const uint64_t b = smem_desc_sw128(kq + (ks >> 2) * TS::HALF + 32 * (ks & 3));
                tc_mma(tbase + C_Z, tbase + C_SL + 8 * ks, b, idesc_bf16(CK), ks > 0);
                tc_mma(tbase + C_Z, tbase + C_SH + 8 * ks, b, idesc_bf16(CK), true);
            }
            tc_commit(bar_z);
            const uint32_t qh = kq + 2 * TS::HALF;
#pragma unroll
            for (int ks = 0; ks < CD / 16; ++ks) {
                const uint64_t b = smem_desc_sw128(qh + (ks >> 2) * TS::HALF + 32 * (ks & 3));
                tc_mma(tbase + C_Y, tbase + C_SL + 8 * ks, b, idesc_bf16(CK), ks > 0);
                tc_mma(tbase + C_Y, tbase + C_SH + 8 * ks, b, idesc_bf16(CK), true);
            }

            if (!mbar_wait(bar_eready, (uint32_t)(ci & 1))) {
                report(p.err, GDN_DEVERR_TIMEOUT);
                break;
            }
            tc_after_sync();
            const uint32_t th = sm_addr(PBc + PW::TH), tl = sm_addr(PBc + PW::TL);
#pragma unroll
            for (int ks = 0; ks < CK / 16; ++ks) {
                const uint64_t bh = smem_desc(th + 256 * ks, (CK / 8) * 128);
                const uint64_t bl = smem_desc(tl + 256 * ks, (CK / 8) * 128);
                tc_mma(tbase + C_U, tbase + C_EL + 8 * ks, bh, idesc_bf16(CK), ks > 0);
                tc_mma(tbase + C_U, tbase + C_EH + 8 * ks, bl, idesc_bf16(CK), true);
                tc_mma(tbase + C_U, tbase + C_EH + 8 * ks, bh, idesc_bf16(CK), true);
            }
            tc_commit(bar_u);

            if (!mbar_wait(bar_wready, (uint32_t)(ci & 1))) {
                report(p.err, GDN_DEVERR_TIMEOUT);
                break;
            }
            tc_after_sync();
            const uint32_t ph = sm_addr(PBc + PW::PH), pl = sm_addr(PBc + PW::PL);
            const uint32_t kt = sm_addr(KT + (ci & 1) * TS::KT_BYTES);
#pragma unroll
            for (int ks = 0; ks < CK / 16; ++ks) {
                const uint64_t b = smem_desc(kt + 256 * ks, (CK / 8) * 128);
                tc_mma(tbase + C_S, tbase + C_WL + 8 * ks, b, idesc_bf16(CD), true);
                tc_mma(tbase + C_S, tbase + C_WH + 8 * ks, b, idesc_bf16(CD), true);
            }
            tc_commit(bar_s);
#pragma unroll
            for (int ks = 0; ks < CK / 16; ++ks) {
                const uint64_t bh = smem_desc(ph + 256 * ks, (CK / 8) * 128);
                const uint64_t bl = smem_desc(pl + 256 * ks, (CK / 8) * 128);
                tc_mma(tbase + C_U, tbase + C_UL + 8 * ks, bh, idesc_bf16(CK), true);
                tc_mma(tbase + C_U, tbase + C_UH + 8 * ks, bl, idesc_bf16(CK), true);
                tc_mma(tbase + C_U, tbase + C_UH + 8 * ks, bh, idesc_bf16(CK), true);
            }
            tc_commit(bar_o);
        }
        __syncwarp(); // lanes 1-31 waited here for lane 0's products
    } else {
        // ======================== loader warp ========================
        // Chunk ci + 1's q, k and v into the buffers of its parity, as soon as
        // their last readers are done: chunk ci - 1's Z and Y products (K | Q)
        // and its E (v), both before its U product's commit (chunk 0's were
        // issued before the wait for the prep kernel).
        // It also stores each chunk's outputs but the last: the compute warps
        // put chunk ci - 1's into the shared tile before they signal chunk
        // ci's E, and wait for this warp's "tile free" before the next fill.
        int issued = 0; // chunks whose copies went out (chunk 0's before the loop)
#pragma unroll 1
        for (int c0 = 0; c0 < L; c0 += CK) {
            const int ci = c0 / CK;
            bool late = false;
            if (c0 + CK < L) {
                if (lane == 0) {
                    late = ci > 0 && !mbar_wait(bar_u, (uint32_t)((ci - 1) & 1));
                    if (!late) {
                        load_chunk(c0 + CK, (ci + 1) & 1);
                        issued = ci + 1;
                    }
                }
                late = __shfl_sync(0xffffffffu, late, 0);
            }
            // every phase of E's barrier, chunk 0's too: a parity wait passes
            // at once on a barrier still a phase behind
            if (!late)
                late = !__all_sync(0xffffffffu, mbar_wait(bar_eready, (uint32_t)(ci & 1)));
            if (late) {
                if (lane == 0)
                    report(p.err, GDN_DEVERR_TIMEOUT);
                break;
            }
            if (ci > 0) {
                store_outputs(c0 - CK, CK, lane, 32); // a chunk before the last is whole
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_osfree);
            }
        }
        // no copy may still be landing when the CTA ends (the compute warps
        // waited for every one unless they stopped early)
        if (lane == 0 && L > 0)
            mbar_wait(bar_in[issued & 1], (uint32_t)((issued >> 1) & 1));
        __syncwarp();
    }

    cp_async_wait_all(); // a chain that stopped early may have the next chunk's inputs in flight
    if (warp < TCC_WARPS)
        tst_wait(); // and S's scaled rows, if it stopped in the wait for U's product
    tc_before_sync();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols) : "memory");
}

} // namespace

size_t prefill_chunked_workspace_bytes(int nseq, int total_tokens, int hv)
{
    if (nseq <= 0 || total_tokens < 0 || hv <= 0)
        return 0;
    return (size_t)prep_units(nseq, total_tokens) * (size_t)hv * (size_t)PW::BYTES;
}

namespace {

// cuTensorMapEncodeTiled, found once through the runtime (no link to the
// driver library)
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// a bf16 [tokens][heads][CD] tensor, boxes of box_inner x 1 head x CK tokens
bool encode_map(CUtensorMap *m, const void *base, int heads, int tokens, int box_inner, bool swizzle128)
{
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)CD, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)CD * 2, (cuuint64_t)heads * CD * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_inner, 1u, (cuuint32_t)CK};
    const cuuint32_t step[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, step,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

} // namespace

cudaError_t launch_gdn_prefill_chunked_tc(const PrefillArgs &a, cudaStream_t s)
{
    const long long ctas = (long long)a.nseq * a.hv;
    if (ctas == 0)
        return cudaSuccess;
    const long long units = prep_units(a.nseq, a.total_tokens);
    if (ctas > 0x7fffffffll || units * a.hv > 0x7fffffffll)
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> configured{0}; // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gdn_chunked_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             TS::TOTAL);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PS::TOTAL);
        // five prep CTAs an SM take more shared memory than the default split leaves
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    // the tensor maps of q, k and v (unused, and left zero, without tokens),
    // before either kernel goes out
    ChunkMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (a.total_tokens > 0 &&
        (!encode_map(&maps.q, a.q, a.hk, a.total_tokens, 64, true) ||
         !encode_map(&maps.k, a.k, a.hk, a.total_tokens, 64, true) ||
         !encode_map(&maps.v, a.v, a.hv, a.total_tokens, CD, false)))
        return cudaErrorInvalidValue;
    unsigned char *work = static_cast<unsigned char *>(a.work);
    cudaError_t e = launch_pdl(gdn_chunk_prep_kernel, dim3((unsigned)(units * a.hv)), dim3(TC_THREADS),
                               (size_t)PS::TOTAL, s, a, work, (int)units);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(gdn_chunked_tc_kernel, dim3((unsigned)ctas), dim3(TCW_THREADS), (size_t)TS::TOTAL, s, a,
                      static_cast<const unsigned char *>(work), (int)units, maps);
}

} // namespace gdn
