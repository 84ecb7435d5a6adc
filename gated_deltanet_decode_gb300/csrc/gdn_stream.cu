// Gated DeltaNet decode, the state kernels (gdn_decode_step and the fused
// conv + GDN layer) as one persistent, warp-specialised TMA pipeline for
// sm_103a.
//
// The step is state traffic: every real (row, value head) reads a dv x dk
// fp32 state and writes the next one, with a few multiply-adds per element
// ("mstar PR #1139", section "Why": a kernel with the same reads and writes
// and no math takes 45.2 of the rule's 46.1 us).  The kernel keeps as many
// bytes in flight as shared memory allows and spends as few instructions as
// it can per byte, since with the memory stream saturated the SMs' issue
// rate is the next limit:
//
//  * Work item = RB consecutive value rows of one (row, value head): 16 KiB of
//    fp32 state (RB = 4096 / dk), contiguous in the pool.  A persistent grid
//    (three CTAs per SM for the fused layer, two for the plain step) splits
//    the items into contiguous ranges, equal to within one item.  With a
//    dozen or more items a CTA, only the first half is split that way; the
//    rest is claimed at run time, a (row, value head) a claim, from a counter
//    the state pool handle owns, so that CTAs on SMs that stream slower take
//    less of the tail (SMs' streaming rates differ by about a fifth).  The
//    last producer to finish resets the counter (and, when asked, commits
//    the slot tables, or stops at a device-side row count for a bucket).
//  * Chains: consecutive items of a CTA that share a row and qk head form a
//    chain.  Only a chain's first item copies q and k (or their conv inputs)
//    and computes the q/k values, their norms and k^ . q^; the rest of the
//    chain reuses them (values in a double-buffered shared buffer, norms in
//    registers).
//  * Producer warp: prepares items 32 at a time (one lane each: slots, gate
//    inputs, gates); one lane streams them: it waits for the item's stage,
//    issues cp.async.bulk copies of the state chunk and of the item's small
//    inputs with their byte count (the first of two arrivals on the stage's
//    "full" mbarrier) and writes the item's metadata (the second).  The first
//    stages' copies leave before the gates are even computed.
//  * v warp (fused layer): computes the item's v channels (conv, one channel
//    a lane) and writes their windows, then signals the stage's "vready".
//  * Consumer warps (8): on a chain's first item, one q or k channel a thread
//    (the conv in the fused layer) and a CTA-wide sum of squares, synchronised
//    by an mbarrier.  Then each lane owns 16 floats of one state row (dk/16
//    lanes a row, 16-byte vectors interleaved so a warp store covers whole
//    128-byte lines), forms u = S k and w = S q with packed f32x2 FMAs and one
//    butterfly, and stores S' = alpha S + c k^ (c = beta (v - alpha u k^))
//    straight to HBM, with o = alpha w + c (k^ . q^).  A warp releases the
//    stage ("empty") as soon as its state row and v are in registers, before
//    the math and the stores.
//  * Every wait is bounded: a wait that runs out reports GDN_DEVERR_TIMEOUT
//    and its warp leaves the loop (no hardware barrier inside the loop can be
//    left waiting); the CTA stops after the producer has waited (bounded) for
//    its copies still in flight.
//
// Fused layer, in place: the q/k conv window of a qk group must be written
// once, after every reader has read it.  With the pool's in-place counters
// (one per slot and qk head, zero between launches) the items are spread
// over the CTAs as in a twin launch, and the v warp counts every item of a
// (slot, qk head) on that pair's counter once the item's copies have landed;
// the item that brings the count to group * chunks comes after every read of
// the old window, so its v warp writes the new window (kept from its chain's
// first item, beside the ring) and sets the counter back to zero.  Without
// the counters (or where that copy does not fit beside the ring) in-place
// launches split the items into ranges of whole groups (all value heads and
// row chunks sharing the qk head), so a group's items run in order on one CTA
// and only the first of them copies and reads the window; it writes the new
// window right after.  Twin launches write another slot, so the chunk-0 item
// of the group's first value head writes it.  The arithmetic per row is the
// same in every schedule, so twin and in place give bit-identical values.
#include <atomic>

#include "gdn_device.cuh"
#include "gdn_ptx.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr float kL2Eps = 1e-6f;
constexpr int kMaxStages = 8;
constexpr int kClaimMinItemsPerCta = 12;

// warps 0-7 consume, warp 8 produces, warp 9 computes v (fused layer only)
template <bool LAYER> constexpr int threads_for() { return kConsumers + 32 + (LAYER ? 32 : 0); }
// CTAs per SM: the fused layer's conv work hides better with more warps; the
// plain step streams better with deeper rings (measured).
template <bool LAYER> constexpr int ctas_per_sm() { return LAYER ? 3 : 2; }

template <int DK> struct Geo {
    static_assert(DK >= 16 && DK <= 256 && DK % 16 == 0, "dk");
    static constexpr int LPR = DK / 16;              // lanes per state row
    static constexpr int RPW = 32 / LPR;             // state rows per warp
    static constexpr int RB = RPW * kConsumerWarps;  // state rows per item (4096 / DK)
};

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
    // raw inputs (bulk-copy destinations)
    // step:  q[DK] | k[DK] | v[RB]
    // layer: win[W-1][NCH] | x[NCH] | w[NCH][W] | bias[NCH], each [q | k | v]
    static constexpr int RAW = STATE + STATE_BYTES;
    static constexpr int WIN = RAW;
    static constexpr int XS = LAYER ? WIN + (W - 1) * NCH * E : RAW;
    static constexpr int WS = XS + NCH * E;
    static constexpr int BS = WS + NCH * W * E;
    static constexpr int RAW_END = LAYER ? BS + NCH * E : RAW + NCH * E;
    static constexpr int VN = align16(RAW_END);                  // v values (fp32) [RB], layer only
    static constexpr int META = align16(VN + (LAYER ? RB * 4 : 0)); // Meta, by the producer
    static constexpr int BYTES = (META + 64 + 127) & ~127;
};

struct Meta {
    int r, h, chunk, rs, ws, live, rows;
    int reuse; // same row and qk head as the previous item: q/k values reused
    float alpha, beta;
};

// Items in (row, value head, chunk) order, which is also (row, qk head,
// value head of the group, chunk): a qk group's items are consecutive.  A
// unit is per_unit consecutive items (per_unit divides hv * chunks); coarse
// launches (in place without counters) take a whole qk group a unit.  The
// first n_static units are split into contiguous ranges, CTA b of g taking
// [first(b), first(b + 1)) (equal to within one unit); the rest are claimed
// `claim` units at a time from the pool's work counter by whichever CTA runs
// out first, so that CTAs that stream slower take less of the tail.
struct Sched {
    int hv, group, chunks;
    int n_units;
    int per_unit;    // items a unit
    int coarse;      // in place, whole qk groups a CTA, the group's first item writes its window
    int n_static;    // units split statically (n_units: no claims)
    int claim;       // units per claim

    __device__ __forceinline__ int first(int b, int g) const
    {
        return (int)(((long long)n_static * b) / g);
    }
    // item i of the whole launch
    __device__ __forceinline__ void item_at(int i, int &r, int &h, int &chunk) const
    {
        chunk = i % chunks;
        const int rh = i / chunks;
        h = rh % hv;
        r = rh / hv;
    }
};

// Stages a CTA holds: as many as fit beside the other CTAs of its SM.  An
// in-place launch with counters also keeps its current chain's new q/k
// window ([W-1][2 DK] activations) after the ring, where the space left over
// holds it (in-place launches of the shapes where it does not fit take whole
// qk groups a CTA).
template <typename T, int DK, bool LAYER, int W> struct Stages {
    static constexpr int avail = (227 * 1024) / ctas_per_sm<LAYER>() - 4096;
    static constexpr int fit = avail / Stage<T, DK, LAYER, W>::BYTES;
    static constexpr int value = fit > kMaxStages ? kMaxStages : fit;
    static_assert(value >= 2, "a stage ring needs two stages");
    static constexpr int RING = value * Stage<T, DK, LAYER, W>::BYTES;
    static constexpr int QKW = LAYER ? (2 * DK * (W - 1) * (int)sizeof(T) + 127) & ~127 : 0;
    static constexpr bool counted_in_place = LAYER && RING + QKW <= avail;
};

template <typename T, int DK, bool LAYER, int W>
__global__ void __launch_bounds__(threads_for<LAYER>(), ctas_per_sm<LAYER>())
gdn_stream_kernel(const StepArgs p, const Sched sc)
{
    using G = Geo<DK>;
    using L = Stage<T, DK, LAYER, W>;
    constexpr int nst = Stages<T, DK, LAYER, W>::value;
    constexpr int RB = G::RB;
    constexpr int E = L::E;

    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bars[3 * kMaxStages + 1]; // full, empty, vready, qk
    __shared__ __align__(16) float qkbuf[2][2 * DK];         // a chain's q | k values, double-buffered
    __shared__ float part[2][kConsumerWarps][2];             // per-warp sums of q^2 and k^2
    __shared__ Meta table[32];                               // the producer's batch
    __shared__ int abort_flag;
    __shared__ int issued_n, consumed_n;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    auto full_bar = [&](int s) { return sm_addr(&bars[s]); };
    auto empty_bar = [&](int s) { return sm_addr(&bars[kMaxStages + s]); };
    auto vready_bar = [&](int s) { return sm_addr(&bars[2 * kMaxStages + s]); };
    const uint32_t qk_bar = sm_addr(&bars[3 * kMaxStages]);
    auto stage = [&](int s) { return smem + (size_t)s * L::BYTES; };
    auto timeout = [&]() {
        report(p.err, GDN_DEVERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
    };

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(full_bar(s), 2); // copies + metadata
            mbar_init(empty_bar(s), kConsumerWarps + (LAYER ? 1 : 0));
            mbar_init(vready_bar(s), 1);
        }
        mbar_init(qk_bar, kConsumerWarps);
        abort_flag = 0;
        issued_n = 0;
        consumed_n = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    wait_prior_grid(); // barrier set-up overlapped the previous kernel's tail

    const int C = p.channels;
    const int group = p.hv / p.hk;

    if (warp == kConsumerWarps) {
        // =========================== producer ===========================
        // Items are prepared up to 32 at a time, one per lane: its slots and
        // gate inputs (independent loads, in flight together) and then its
        // gates.  One lane streams the batch: for each item it waits for the
        // item's stage, issues the bulk copies with their byte count (the
        // first of two arrivals on "full") and writes the item's metadata (the
        // second).  At the start the first nst items' copies go out as soon as
        // their slots are known, before the gates are computed.  The CTA's
        // static range comes first, then claimed ranges; a metadata-only
        // stage with live = -1 ends the stream.
        int lo = sc.first(blockIdx.x, gridDim.x) * sc.per_unit; // items [lo, hi) to do next
        int hi = sc.first(blockIdx.x + 1, gridDim.x) * sc.per_unit;
        const bool claims = sc.n_static < sc.n_units;
        // a bucket's decode half: rows at or past the device count are not this launch's
        int live_rows = p.rows;
        if (p.n_live) {
            const int nl = *p.n_live;
            live_rows = nl < 0 ? 0 : (nl < p.rows ? nl : p.rows);
        }
        const bool counted = claims || p.commit; // producers count themselves done
        int kdone = 0;                // items issued so far
        int prev_r = -1, prev_g = -1; // the item before the batch
        bool stop = false;

        // issue item k's copies into its stage (first arrival on "full")
        auto issue = [&](int k, const Meta &q) -> bool {
            const int s = k % nst;
            if (!mbar_wait(empty_bar(s), (uint32_t)((k / nst) & 1) ^ 1u)) {
                timeout();
                return false;
            }
            if (*(volatile int *)&abort_flag)
                return false;
            unsigned char *st = stage(s);
            const uint32_t fb = full_bar(s);
            if (!q.live) {
                mbar_arrive(fb);
                return true;
            }
            const int r = q.r, h = q.h, chunk = q.chunk, rows = q.rows;
            const int g = h / group;
            const int cq = g * DK, ck = p.hk * DK + g * DK;
            const int cv = 2 * p.hk * DK + h * p.dv + chunk * RB;
            const int nqk = q.reuse ? 0 : 2 * DK; // q/k channels to copy
            uint32_t bytes = (uint32_t)(rows * DK * 4);
            if constexpr (LAYER)
                bytes += (uint32_t)(((W - 1) + 1 + W + (p.bias ? 1 : 0)) * (nqk + rows) * E);
            else
                bytes += (uint32_t)((nqk + rows) * E);
            mbar_arrive_tx(fb, bytes);
            const float *src = p.pool + (((size_t)q.rs * p.hv + h) * p.dv + (size_t)chunk * RB) * DK;
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
                    if (sgm < 2 && q.reuse)
                        continue;
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
                if (!q.reuse) {
                    bulk_load(sm_addr(st + L::RAW), qp + ((size_t)r * p.hk + g) * DK * E, DK * E, fb);
                    bulk_load(sm_addr(st + L::RAW + DK * E), kp + ((size_t)r * p.hk + g) * DK * E, DK * E, fb);
                }
                bulk_load(sm_addr(st + L::RAW + 2 * DK * E),
                          vp + (((size_t)r * p.hv + h) * p.dv + (size_t)chunk * RB) * E, (uint32_t)(rows * E), fb);
            }
            return true;
        };
        // write item k's metadata (second arrival on "full")
        auto publish = [&](int k, const Meta &q) {
            unsigned char *st = stage(k % nst);
            *reinterpret_cast<Meta *>(st + L::META) = q;
            mbar_arrive(full_bar(k % nst));
            issued_n = k + 1;
        };

        while (!stop) {
            if (lo >= hi) {
                if (!claims)
                    break;
                int u = 0;
                if (lane == 0)
                    u = (int)atomicAdd(p.work, (unsigned)sc.claim);
                u = __shfl_sync(0xffffffffu, u, 0) + sc.n_static;
                if (u >= sc.n_units)
                    break;
                lo = u * sc.per_unit;
                hi = min(u + sc.claim, sc.n_units) * sc.per_unit;
            }
            const int nb = min(32, hi - lo);
            const int base = kdone;
            const bool valid = lane < nb;
            Meta q;
            q.r = q.h = q.chunk = q.rs = q.ws = q.live = q.rows = q.reuse = 0;
            q.alpha = q.beta = 0.f;
            float av = 0.f, bv = 0.f, al = 0.f, dt = 0.f;
            if (valid) {
                sc.item_at(lo + lane, q.r, q.h, q.chunk);
                if (q.r < live_rows) {
                    q.rs = p.read_slot[q.r];
                    q.ws = p.in_place ? q.rs : p.write_slot[q.r];
                }
                av = ld_act<T>(p.a, (size_t)q.r * p.hv + q.h);
                bv = ld_act<T>(p.b, (size_t)q.r * p.hv + q.h);
                al = p.A_log[q.h];
                dt = p.dt_bias[q.h];
            }
            const int g = q.h / group;
            int pr = __shfl_up_sync(0xffffffffu, q.r, 1), pg = __shfl_up_sync(0xffffffffu, g, 1);
            if (lane == 0) {
                pr = prev_r;
                pg = prev_g;
            }
            prev_r = __shfl_sync(0xffffffffu, q.r, nb - 1);
            prev_g = __shfl_sync(0xffffffffu, g, nb - 1);
            if (valid) {
                const int cls = classify_row(q.rs, q.ws, p.num_slots, p.in_place != 0);
                if (cls < 0)
                    report(p.err, GDN_DEVERR_BAD_SLOT);
                q.live = cls == 1;
                q.rows = min(RB, p.dv - q.chunk * RB);
                // a chain continues only through live items (liveness is per row)
                q.reuse = q.live && pr == q.r && pg == g;
            }
            table[lane] = q; // everything but the gates
            __syncwarp();
            // start-up: the first stages' copies go out before the gates are computed
            const int early = base == 0 ? min(nst, nb) : 0;
            if (lane == 0) {
                for (int j = 0; j < early; ++j)
                    if (!issue(j, table[j])) {
                        stop = true;
                        break;
                    }
            }
            if (q.live) {
                table[lane].alpha = gate_alpha(al, av, dt);
                table[lane].beta = gate_beta(bv);
            }
            __syncwarp();
            if (lane == 0 && !stop) {
                for (int j = 0; j < early; ++j)
                    publish(base + j, table[j]);
                for (int j = early; j < nb; ++j) {
                    const Meta qq = table[j];
                    if (!issue(base + j, qq)) {
                        stop = true;
                        break;
                    }
                    publish(base + j, qq);
                }
            }
            stop = __shfl_sync(0xffffffffu, stop, 0);
            __syncwarp();
            kdone += nb;
            lo += nb;
        }
        // This CTA makes no more claims and reads no more slots.  The last CTA
        // to get here (every other one has counted itself done after its last
        // claim and its last slot load) commits the slot tables if asked and
        // resets the counters for the pool's next launch.
        if (counted) {
            int last = 0;
            if (lane == 0) {
                // release: this producer's slot loads come before its count;
                // acquire: the last one's writes come after every other's loads
                unsigned done;
                asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                             : "=r"(done)
                             : "l"(p.work + 1)
                             : "memory");
                last = done == gridDim.x - 1;
            }
            if (__shfl_sync(0xffffffffu, last, 0)) {
                if (p.commit) {
                    // the whole warp swaps the tables, 256 rows a round, loads first
                    int32_t *rs = const_cast<int32_t *>(p.read_slot);
                    int32_t *ws = const_cast<int32_t *>(p.write_slot);
                    for (int r0 = 0; r0 < live_rows; r0 += 256) {
                        int32_t vr[8], vw[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int r = r0 + 32 * j + lane;
                            if (r < live_rows) {
                                vr[j] = rs[r];
                                vw[j] = ws[r];
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int r = r0 + 32 * j + lane;
                            if (r < live_rows) {
                                rs[r] = vw[j];
                                ws[r] = vr[j];
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    atomicExch(p.work, 0u);
                    atomicExch(p.work + 1, 0u);
                }
            }
        }
        // end of the stream
        if (lane == 0 && !stop) {
            const int s = kdone % nst;
            if (!mbar_wait(empty_bar(s), (uint32_t)((kdone / nst) & 1) ^ 1u)) {
                timeout();
            } else {
                Meta e;
                e.r = e.h = e.chunk = e.rs = e.ws = e.rows = e.reuse = 0;
                e.live = -1;
                e.alpha = e.beta = 0.f;
                *reinterpret_cast<Meta *>(stage(s) + L::META) = e;
                mbar_arrive(full_bar(s)); // both arrivals: no copies
                mbar_arrive(full_bar(s));
                issued_n = kdone + 1;
            }
        }
    } else if (LAYER && warp == kConsumerWarps + 1) {
        // =========================== v warp =============================
        if constexpr (LAYER) {
            // In place with counters: the count of item k goes out after its
            // stage is released and is looked at (settled) one item later, or
            // before a new chain overwrites the kept window, so its latency hides
            // behind the next item's wait.  A lane keeps the channels c = lane +
            // 32 i of the window, written and read by that lane alone.
            const bool counted_ip = p.in_place && !sc.coarse;
            const unsigned per_pair = (unsigned)(group * sc.chunks);
            T *qkw = reinterpret_cast<T *>(smem + Stages<T, DK, LAYER, W>::RING); // [W-1][2 DK]
            unsigned *pend = nullptr; // the counter whose count is in flight
            unsigned pend_old = 0;    // lane 0: the value before that count
            int pend_slot = 0, pend_g = 0;
            auto settle = [&]() {
                if (!pend)
                    return;
                const unsigned old = __shfl_sync(0xffffffffu, pend_old, 0);
                if (old == per_pair - 1) {
                    // every item of the pair has counted, so every read of the old window is done
                    T *wout = reinterpret_cast<T *>(p.conv) + (size_t)pend_slot * (W - 1) * C;
                    for (int c = lane; c < 2 * DK; c += 32) {
                        const int gc = c < DK ? pend_g * DK + c : p.hk * DK + pend_g * DK + (c - DK);
#pragma unroll
                        for (int j = 0; j < W - 1; ++j)
                            wout[(size_t)j * C + gc] = qkw[j * 2 * DK + c];
                    }
                    if (lane == 0)
                        atomicExch(pend, 0u); // zero for the pool's next launch
                }
                pend = nullptr;
            };
            for (int k = 0;; ++k) {
                const int s = k % nst;
                if (!mbar_wait(full_bar(s), (uint32_t)((k / nst) & 1))) {
                    timeout();
                    break;
                }
                unsigned char *st = stage(s);
                const Meta m = *reinterpret_cast<const Meta *>(st + L::META);
                if (m.live < 0) {
                    settle();
                    break; // end of the stream
                }
                if (counted_ip && m.live && !m.reuse) {
                    // a chain starts: keep its new q/k window (old positions 1..W-2, then x)
                    settle();
                    const T *win = reinterpret_cast<const T *>(st + L::WIN);
                    const T *xs = reinterpret_cast<const T *>(st + L::XS);
                    for (int c = lane; c < 2 * DK; c += 32) {
#pragma unroll
                        for (int j = 0; j + 1 < W - 1; ++j)
                            qkw[j * 2 * DK + c] = win[(j + 1) * L::NCH + c];
                        qkw[(W - 2) * 2 * DK + c] = xs[c];
                    }
                }
                if (m.live) {
                    float *vn = reinterpret_cast<float *>(st + L::VN);
                    T *wout = reinterpret_cast<T *>(p.conv) + (size_t)m.ws * (W - 1) * C;
                    for (int c = lane; c < m.rows; c += 32) {
                        float wv[W], winv[W - 1];
#pragma unroll
                        for (int j = 0; j < W; ++j)
                            wv[j] = sh_act<T>(st + L::WS, (2 * DK + c) * W + j);
#pragma unroll
                        for (int j = 0; j < W - 1; ++j)
                            winv[j] = sh_act<T>(st + L::WIN, j * L::NCH + 2 * DK + c);
                        const float xv = sh_act<T>(st + L::XS, 2 * DK + c);
                        const float bv = p.bias ? sh_act<T>(st + L::BS, 2 * DK + c) : 0.f;
                        vn[c] = round_act<T>(conv_channel<W>(winv, xv, wv, bv, p.silu != 0));
                        // this item is the only reader and writer of its v channels
                        const int cv = 2 * p.hk * DK + m.h * p.dv + m.chunk * RB + c;
#pragma unroll
                        for (int j = 0; j + 1 < W - 1; ++j)
                            wout[(size_t)j * C + cv] = from_f<T>(winv[j + 1]);
                        wout[(size_t)(W - 2) * C + cv] = from_f<T>(xv);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(vready_bar(s));
                    mbar_arrive(empty_bar(s));
                }
                if (counted_ip && m.live) {
                    settle();
                    const int g = m.h / group;
                    pend = p.qk_count + (size_t)m.rs * p.qk_stride + g;
                    pend_slot = m.rs;
                    pend_g = g;
                    if (lane == 0)
                        pend_old = atomicAdd(pend, 1u);
                }
            }
        }
    } else if (warp < kConsumerWarps) {
        // =========================== consumers ==========================
        const int lrow = lane / G::LPR, lcol = lane % G::LPR;
        const int t = tid; // consumer index 0..255
        const int row = warp * G::RPW + lrow;
        int chains = 0;                // chains started so far
        int qkb = 0;                   // buffer of the current chain
        float inv_q = 0.f, inv_k = 0.f, kappa = 0.f;
        for (int k = 0;; ++k) {
            const int s = k % nst;
            const uint32_t par = (uint32_t)((k / nst) & 1);
            if (!mbar_wait(full_bar(s), par)) {
                timeout();
                break;
            }
            unsigned char *st = stage(s);
            const Meta m = *reinterpret_cast<const Meta *>(st + L::META);
            if (m.live < 0)
                break; // end of the stream
            T *out = reinterpret_cast<T *>(p.out) + ((size_t)m.r * p.hv + m.h) * p.dv + (size_t)m.chunk * RB;
            if (m.live) {
                if (!m.reuse) {
                    // ---- a chain starts: q/k values, norms, k^ . q^ -----------------
                    qkb = chains & 1;
                    float *qk = qkbuf[qkb];
                    const int g = m.h / group;
                    float psq = 0.f, psk = 0.f;
                    for (int c = t; c < 2 * DK; c += kConsumers) {
                        const bool isq = c < DK;
                        float val;
                        if constexpr (LAYER) {
                            float wq[W], winq[W - 1];
#pragma unroll
                            for (int j = 0; j < W; ++j)
                                wq[j] = sh_act<T>(st + L::WS, c * W + j);
#pragma unroll
                            for (int j = 0; j < W - 1; ++j)
                                winq[j] = sh_act<T>(st + L::WIN, j * L::NCH + c);
                            const float xq = sh_act<T>(st + L::XS, c);
                            const float bq = p.bias ? sh_act<T>(st + L::BS, c) : 0.f;
                            val = round_act<T>(conv_channel<W>(winq, xq, wq, bq, p.silu != 0));
                            // The q/k window is written once per group.  Twin: by the chunk-0
                            // item of the group's first value head (it writes another slot).
                            // In place, whole groups a CTA: a group's only window reader is
                            // its first item, which writes the window as soon as its own
                            // copy has landed.  In place with counters: by the v warp of the group's
                            // last item (above), never here.
                            const bool writer =
                                p.in_place ? sc.coarse != 0 : (m.h % group == 0 && m.chunk == 0);
                            if (writer) {
                                T *wout = reinterpret_cast<T *>(p.conv) + (size_t)m.ws * (W - 1) * C;
                                const int gc = isq ? g * DK + c : p.hk * DK + g * DK + (c - DK);
#pragma unroll
                                for (int j = 0; j + 1 < W - 1; ++j)
                                    wout[(size_t)j * C + gc] = from_f<T>(winq[j + 1]);
                                wout[(size_t)(W - 2) * C + gc] = from_f<T>(xq);
                            }
                        } else {
                            val = sh_act<T>(st + L::RAW, c);
                        }
                        qk[c] = val;
                        if (isq)
                            psq = __fmaf_rn(val, val, psq);
                        else
                            psk = __fmaf_rn(val, val, psk);
                    }
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) {
                        psq += __shfl_xor_sync(0xffffffffu, psq, off);
                        psk += __shfl_xor_sync(0xffffffffu, psk, off);
                    }
                    if (lane == 0) {
                        part[qkb][warp][0] = psq;
                        part[qkb][warp][1] = psk;
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(qk_bar);
                    if (!mbar_wait(qk_bar, (uint32_t)(chains & 1))) {
                        timeout();
                        break;
                    }
                    ++chains;
                    float qq = 0.f, kk2 = 0.f;
#pragma unroll
                    for (int wi = 0; wi < kConsumerWarps; ++wi) {
                        qq += part[qkb][wi][0];
                        kk2 += part[qkb][wi][1];
                    }
                    inv_q = __fdiv_rn(1.0f, sqrtf(qq + kL2Eps)) * rsqrtf((float)DK);
                    inv_k = __fdiv_rn(1.0f, sqrtf(kk2 + kL2Eps));
                    float pqk = 0.f;
                    for (int i = lane; i < DK; i += 32)
                        pqk = __fmaf_rn(qk[i], qk[DK + i], pqk);
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        pqk += __shfl_xor_sync(0xffffffffu, pqk, off);
                    kappa = pqk * inv_q * inv_k; // k^ . q^
                }

                // ---- this lane's state row ---------------------------------------
                float vi = 0.f;
                if constexpr (LAYER) {
                    if (!mbar_wait(vready_bar(s), par)) {
                        timeout();
                        break;
                    }
                    if (row < m.rows)
                        vi = reinterpret_cast<const float *>(st + L::VN)[row];
                } else {
                    if (row < m.rows)
                        vi = sh_act<T>(st + L::RAW, 2 * DK + row);
                }
                const float *kq = qkbuf[qkb];
                const float *srow = reinterpret_cast<const float *>(st + L::STATE) + row * DK + 4 * lcol;
                float4 kh[4], qh[4], sv[4];
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    sv[mm] = *reinterpret_cast<const float4 *>(srow + 4 * G::LPR * mm);
                // The warp has all it needs from the stage (state row, v, metadata;
                // q/k values live outside the stages): release it before the math and
                // the stores, so its next copy starts sooner.
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty_bar(s));
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    const int j = 4 * (lcol + G::LPR * mm);
                    qh[mm] = *reinterpret_cast<const float4 *>(&kq[j]);
                    kh[mm] = *reinterpret_cast<const float4 *>(&kq[DK + j]);
                }
                // u = S . k and w = S . q on the raw values; the shuffles need the
                // whole warp, so every lane reduces and only real rows are stored
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
                if (row < m.rows) {
                    const float alpha = m.alpha, beta = m.beta;
                    const float c = beta * __fmaf_rn(-alpha, u, vi);
                    const float o = __fmaf_rn(c, kappa, alpha * wd);
                    const float ck = c * inv_k; // S' = alpha S + c k^ = alpha S + (c / |k|) k
                    const float2 a2 = make_float2(alpha, alpha), c2 = make_float2(ck, ck);
                    float *dst = p.pool +
                                 (((size_t)m.ws * p.hv + m.h) * p.dv + (size_t)m.chunk * RB + row) * DK + 4 * lcol;
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        const float2 lo = fma2(c2, make_float2(kh[mm].x, kh[mm].y),
                                               mul2(a2, make_float2(sv[mm].x, sv[mm].y)));
                        const float2 hi = fma2(c2, make_float2(kh[mm].z, kh[mm].w),
                                               mul2(a2, make_float2(sv[mm].z, sv[mm].w)));
                        st_state(dst + 4 * G::LPR * mm, make_float4(lo.x, lo.y, hi.x, hi.y));
                    }
                    if (lcol == 0)
                        out[row] = from_f<T>(o);
                }
            } else {
                // padding or bad row: zero outputs, no slot touched
                if (t < m.rows)
                    out[t] = from_f<T>(0.f);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty_bar(s));
            }
            if (t == 0)
                consumed_n = k + 1;
        }
    }

    // A CTA whose waits ran out leaves no copy in flight: the producer waits
    // (bounded) for every stage it filled that was not consumed.
    asm volatile("barrier.sync 0;" ::: "memory"); // warps arrive here at different times
    if (abort_flag && tid == kConsumers) {
        for (int k = consumed_n; k < issued_n; ++k)
            mbar_wait(full_bar(k % nst), (uint32_t)((k / nst) & 1));
    }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
std::atomic<int> g_num_sms[64] = {};

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

// A launch's split: units of per_unit items, the first n_static of them in
// static ranges over `grid` CTAs, the rest claimed `claim` units at a time.
struct Split {
    int per_unit, n_units, grid, n_static, claim;
};

Split make_split(long long items, int per_unit, int chunks, int slots, bool can_claim)
{
    Split p;
    p.per_unit = per_unit;
    p.n_units = (int)(items / per_unit);
    p.grid = p.n_units < slots ? p.n_units : slots;
    // With a dozen or more items a CTA, half of the units are claimed at run
    // time, about a (row, value head) a claim; with fewer, the claims' latency
    // costs more than the balance they buy (measured on the 0.8B and 9B layer
    // shapes at 16 to 256 rows).
    p.claim = (chunks < 4 ? chunks : 4) / per_unit;
    if (p.claim < 1)
        p.claim = 1;
    p.n_static = p.n_units;
    if (can_claim && items >= (long long)kClaimMinItemsPerCta * p.grid)
        p.n_static = p.n_units / 2 / p.claim * p.claim;
    return p;
}

// The longest share of a CTA under a split, in item times: the largest
// static range plus one claim, each chain start (q/k conv, norms and their
// CTA-wide sum, once per row and qk head a CTA meets) counted as 1.5 items.
// A static range of single items that cuts chains meets up to one chain more
// than whole chains would.  Fitted on the fused layer (0.8B and 9B shapes,
// 1 to 256 rows, twin and in place): single items at 1-8, 32 and 64 rows of
// the 0.8B shape and at every size of the 9B one (whose chains are 8 items),
// whole chains at 16, 24, 48 and 96 rows of the 0.8B shape (10 % faster at
// 16 and 24 rows); where it picks the slower of the two, by under 0.25 us.
double share_cost(const Split &p, int chain)
{
    if (p.grid <= 0)
        return 0.0;
    const long long m = ((long long)p.n_static + p.grid - 1) / p.grid; // units in the largest range
    const long long it = m * p.per_unit;
    long long starts = p.per_unit >= chain ? m : (it > 0 ? 1 + (it - 1 + chain - 1) / chain : 0);
    if (starts > it)
        starts = it;
    double cost = (double)it + 1.5 * (double)starts;
    if (p.n_static < p.n_units)
        cost += (double)p.claim * p.per_unit + 1.5;
    return cost;
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
    // in place without room for the kept window: whole groups a CTA
    if (LAYER && a.in_place && !Stages<T, DK, LAYER, W>::counted_in_place)
        coarse = true;
    sc.coarse = coarse ? 1 : 0;
    const long long items = (long long)a.rows * a.hv * sc.chunks;
    if (items > (1ll << 30))
        return cudaErrorInvalidValue;
    if (items == 0)
        return cudaSuccess;
    // ctas_per_sm CTAs per SM, each with as many stages as fit
    constexpr int kCtas = ctas_per_sm<LAYER>();
    const int slots = kCtas * num_sms();
    // a unit: one item, or a whole chain (a row's qk group: group value heads
    // x chunks), whichever gives the shorter longest share; coarse launches
    // take whole chains
    const int chain = sc.group * sc.chunks;
    Split sp = make_split(items, coarse ? chain : 1, sc.chunks, slots, a.work != nullptr);
    if (!coarse) {
        const Split whole = make_split(items, chain, sc.chunks, slots, a.work != nullptr);
        if (share_cost(whole, chain) < share_cost(sp, chain))
            sp = whole;
    }
    sc.per_unit = sp.per_unit;
    sc.n_units = sp.n_units;
    sc.n_static = sp.n_static;
    sc.claim = sp.claim;
    using ST = Stages<T, DK, LAYER, W>;
    const size_t smem_max = (size_t)ST::RING + (ST::counted_in_place ? ST::QKW : 0);
    const size_t smem = (size_t)ST::RING + (LAYER && a.in_place && !coarse ? ST::QKW : 0);
    auto kern = gdn_stream_kernel<T, DK, LAYER, W>;
    static std::atomic<unsigned long long> configured{0}; // one bit per device, per instantiation
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
        if (e != cudaSuccess)
            return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    return launch_pdl(kern, dim3(sp.grid), dim3(threads_for<LAYER>()), smem, s, a, sc);
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
    const bool coarse = a.in_place != 0 && a.qk_count == nullptr;
    switch (a.width) {
    case 2: return dtype == GDN_BF16 ? dispatch_dk<__nv_bfloat16, true, 2>(a, coarse, s) : dispatch_dk<float, true, 2>(a, coarse, s);
    case 3: return dtype == GDN_BF16 ? dispatch_dk<__nv_bfloat16, true, 3>(a, coarse, s) : dispatch_dk<float, true, 3>(a, coarse, s);
    case 4: return dtype == GDN_BF16 ? dispatch_dk<__nv_bfloat16, true, 4>(a, coarse, s) : dispatch_dk<float, true, 4>(a, coarse, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gdn
