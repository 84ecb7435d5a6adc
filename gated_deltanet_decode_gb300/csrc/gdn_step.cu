// Gated DeltaNet decode: the state kernels (gdn_decode_step and the fused
// conv + GDN layer), sm_103a.
//
// The step is state traffic: every real (row, value head) reads a dv x dk
// fp32 state and writes the next one, and the arithmetic per state element is
// two multiply-adds for the reductions and one for the update ("mstar PR
// #1139", section "Why": a kernel with the same reads and writes and no math
// takes 45.2 of the rule's 46.1 us).  So the kernel is built around the
// stream:
//
//  * A block owns RB consecutive value rows of one (row, value head): a
//    chunk of the head's state, RB * dk * 4 bytes, read once and written once.
//  * Within a block, LPR = dk/16 lanes own one state row; a lane holds 16
//    floats of it as four 16-byte vectors, interleaved so that each vector
//    load of the warp covers whole 128-byte lines.
//  * The state loads are issued first; the prologue (q/k normalisation, the
//    gates, and in the fused layer the causal conv of the block's channels)
//    runs while they are in flight.
//  * Per state row i the two reductions u_i = S_i . k^ and w_i = S_i . q^
//    share one butterfly over the LPR lanes; then
//        c_i  = beta (v_i - alpha u_i)
//        S'_i = alpha S_i + c_i k^          (= alpha S_i (I - beta k^ k^T) + beta v_i k^T)
//        o_i  = alpha w_i + c_i (k^ . q^)   (= S'_i . q^)
//    and S'_i goes straight back out.
//
// Fused layer, in-place mode: the conv window of the q/k channels is read by
// every block of the qk head's group (all value heads sharing the qk head, all
// row chunks) and written once.  Those blocks form one thread-block cluster;
// each arrives on the cluster barrier after reading the window and the
// designated writer waits on it before overwriting the window.  In twin mode
// the window is written to another slot and no cluster is needed.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kL2Eps = 1e-6f;

template <int DK> struct Geo {
    static_assert(DK >= 16 && DK <= 256 && DK % 16 == 0, "dk");
    static constexpr int LPR = DK / 16;      // lanes per state row
    static constexpr int RPW = 32 / LPR;     // state rows per warp per pass
    static constexpr int RPB = RPW * kWarps; // state rows per block per pass
};

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

template <typename T>
__device__ __forceinline__ float load_act(const void *base, size_t idx)
{
    return to_f(reinterpret_cast<const T *>(base)[idx]);
}

// One launch = one of:
//   LAYER = false: gdn_decode_step (q, k, v given)
//   LAYER = true : conv + rule; CLUSTER = true for in-place mode.
template <typename T, int DK, int PASSES, bool LAYER, int W, bool CLUSTER>
__global__ void __launch_bounds__(kThreads) gdn_state_kernel(const StepArgs p, int chunks)
{
    using G = Geo<DK>;
    constexpr int RB = G::RPB * PASSES; // value rows per block
    static_assert(RB <= kThreads, "one v channel per thread in the prologue");

    __shared__ __align__(16) float sh_q[DK];
    __shared__ __align__(16) float sh_k[DK];
    __shared__ float sh_v[RB];
    __shared__ float sh_part[3][kWarps];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int lrow = lane / G::LPR, lcol = lane % G::LPR;
    const int chunk = blockIdx.x % chunks;
    const int rh = blockIdx.x / chunks;
    const int h = rh % p.hv;
    const int r = rh / p.hv;
    const int group = p.hv / p.hk;
    const int g = h / group;

    const int rs = p.read_slot[r];
    const int ws = p.in_place ? rs : p.write_slot[r];
    const int cls = classify_row(rs, ws, p.num_slots, p.in_place != 0);
    if (cls < 0 && tid == 0)
        report(p.err, GDN_DEVERR_BAD_SLOT);
    const bool live = cls == 1;

    const size_t head_elems = (size_t)p.dv * DK;
    const float *Sin = p.pool + ((size_t)(live ? rs : 0) * p.hv + h) * head_elems;
    float *Sout = p.pool + ((size_t)(live ? ws : 0) * p.hv + h) * head_elems;

    // ---- 1. issue the state loads ------------------------------------
    float4 s[PASSES][4];
    int srow[PASSES];
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
        srow[ps] = chunk * RB + ps * G::RPB + warp * G::RPW + lrow;
        if (live && srow[ps] < p.dv) {
            const float *src = Sin + (size_t)srow[ps] * DK + 4 * lcol;
#pragma unroll
            for (int m = 0; m < 4; ++m)
                s[ps][m] = ld_state(src + 4 * G::LPR * m);
        }
    }

    // ---- 2. prologue: q, k, v (from the conv in the fused layer) -------
    float part_qq = 0.f, part_kk = 0.f, part_qk = 0.f;
    // q/k window of this thread's channel, kept for the deferred write
    float keep_q[W], keep_k[W];
    (void)keep_q;
    (void)keep_k;
    const bool writer = LAYER && (h % group == 0) && chunk == 0;
    if (live) {
        if (tid < DK) {
            float qv, kv;
            if constexpr (LAYER) {
                const int C = p.channels;
                const int cq = g * DK + tid;
                const int ck = p.hk * DK + g * DK + tid;
                const size_t win_in = (size_t)rs * (W - 1) * C;
                float wq[W], wk[W], winq[W - 1], wink[W - 1];
#pragma unroll
                for (int j = 0; j < W; ++j) {
                    wq[j] = load_act<T>(p.w, (size_t)cq * W + j);
                    wk[j] = load_act<T>(p.w, (size_t)ck * W + j);
                }
#pragma unroll
                for (int j = 0; j < W - 1; ++j) {
                    winq[j] = load_act<T>(p.conv, win_in + (size_t)j * C + cq);
                    wink[j] = load_act<T>(p.conv, win_in + (size_t)j * C + ck);
                }
                const float xq = load_act<T>(p.x, (size_t)r * C + cq);
                const float xk = load_act<T>(p.x, (size_t)r * C + ck);
                const float bq = p.bias ? load_act<T>(p.bias, cq) : 0.f;
                const float bk = p.bias ? load_act<T>(p.bias, ck) : 0.f;
                qv = round_act<T>(conv_channel<W>(winq, xq, wq, bq, p.silu != 0));
                kv = round_act<T>(conv_channel<W>(wink, xk, wk, bk, p.silu != 0));
#pragma unroll
                for (int j = 0; j + 1 < W - 1; ++j) {
                    keep_q[j] = winq[j + 1];
                    keep_k[j] = wink[j + 1];
                }
                keep_q[W - 2] = xq;
                keep_k[W - 2] = xk;
                if (!CLUSTER && writer) {
                    T *wout = reinterpret_cast<T *>(p.conv) + (size_t)ws * (W - 1) * C;
#pragma unroll
                    for (int j = 0; j < W - 1; ++j) {
                        wout[(size_t)j * C + cq] = from_f<T>(keep_q[j]);
                        wout[(size_t)j * C + ck] = from_f<T>(keep_k[j]);
                    }
                }
            } else {
                qv = load_act<T>(p.q, ((size_t)r * p.hk + g) * DK + tid);
                kv = load_act<T>(p.k, ((size_t)r * p.hk + g) * DK + tid);
            }
            sh_q[tid] = qv;
            sh_k[tid] = kv;
            part_qq = qv * qv;
            part_kk = kv * kv;
            part_qk = qv * kv;
        }
        if (tid < RB) {
            const int i = chunk * RB + tid;
            if (i < p.dv) {
                float vv;
                if constexpr (LAYER) {
                    const int C = p.channels;
                    const int cv = 2 * p.hk * DK + h * p.dv + i;
                    const size_t win_in = (size_t)rs * (W - 1) * C;
                    float wv[W], winv[W - 1];
#pragma unroll
                    for (int j = 0; j < W; ++j)
                        wv[j] = load_act<T>(p.w, (size_t)cv * W + j);
#pragma unroll
                    for (int j = 0; j < W - 1; ++j)
                        winv[j] = load_act<T>(p.conv, win_in + (size_t)j * C + cv);
                    const float xv = load_act<T>(p.x, (size_t)r * C + cv);
                    const float bv = p.bias ? load_act<T>(p.bias, cv) : 0.f;
                    vv = round_act<T>(conv_channel<W>(winv, xv, wv, bv, p.silu != 0));
                    // this block is the only reader and writer of channel cv
                    T *wout = reinterpret_cast<T *>(p.conv) + (size_t)ws * (W - 1) * C;
#pragma unroll
                    for (int j = 0; j + 1 < W - 1; ++j)
                        wout[(size_t)j * C + cv] = from_f<T>(winv[j + 1]);
                    wout[(size_t)(W - 2) * C + cv] = from_f<T>(xv);
                } else {
                    vv = load_act<T>(p.v, ((size_t)r * p.hv + h) * p.dv + i);
                }
                sh_v[tid] = vv;
            }
        }
    }
    if constexpr (CLUSTER)
        cluster_arrive_release(); // this block has read its conv windows

    // block reduction of |q|^2, |k|^2, q.k (fixed order: deterministic)
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        part_qq += __shfl_xor_sync(0xffffffffu, part_qq, off);
        part_kk += __shfl_xor_sync(0xffffffffu, part_kk, off);
        part_qk += __shfl_xor_sync(0xffffffffu, part_qk, off);
    }
    if (lane == 0) {
        sh_part[0][warp] = part_qq;
        sh_part[1][warp] = part_kk;
        sh_part[2][warp] = part_qk;
    }
    __syncthreads();

    T *out = reinterpret_cast<T *>(p.out) + ((size_t)r * p.hv + h) * p.dv;
    if (live) {
        float qq = 0.f, kk = 0.f, qk = 0.f;
        constexpr int kRedWarps = (DK + 31) / 32;
#pragma unroll
        for (int wi = 0; wi < kRedWarps; ++wi) {
            qq += sh_part[0][wi];
            kk += sh_part[1][wi];
            qk += sh_part[2][wi];
        }
        const float inv_q = __fdiv_rn(1.0f, sqrtf(qq + kL2Eps)) * rsqrtf((float)DK);
        const float inv_k = __fdiv_rn(1.0f, sqrtf(kk + kL2Eps));
        const float kappa = qk * inv_q * inv_k; // k^ . q^

        const float alpha = gate_alpha(p.A_log[h], load_act<T>(p.a, (size_t)r * p.hv + h), p.dt_bias[h]);
        const float beta = gate_beta(load_act<T>(p.b, (size_t)r * p.hv + h));

        // this lane's slices of k^ and q^
        float4 kh[4], qh[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int j = 4 * (lcol + G::LPR * m);
            const float4 kr = *reinterpret_cast<const float4 *>(&sh_k[j]);
            const float4 qr = *reinterpret_cast<const float4 *>(&sh_q[j]);
            kh[m] = make_float4(kr.x * inv_k, kr.y * inv_k, kr.z * inv_k, kr.w * inv_k);
            qh[m] = make_float4(qr.x * inv_q, qr.y * inv_q, qr.z * inv_q, qr.w * inv_q);
        }

#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int i = srow[ps];
            const bool valid = i < p.dv;
            float u = 0.f, wdot = 0.f;
            if (valid) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    u = __fmaf_rn(s[ps][m].x, kh[m].x, u);
                    u = __fmaf_rn(s[ps][m].y, kh[m].y, u);
                    u = __fmaf_rn(s[ps][m].z, kh[m].z, u);
                    u = __fmaf_rn(s[ps][m].w, kh[m].w, u);
                    wdot = __fmaf_rn(s[ps][m].x, qh[m].x, wdot);
                    wdot = __fmaf_rn(s[ps][m].y, qh[m].y, wdot);
                    wdot = __fmaf_rn(s[ps][m].z, qh[m].z, wdot);
                    wdot = __fmaf_rn(s[ps][m].w, qh[m].w, wdot);
                }
            }
#pragma unroll
            for (int off = G::LPR / 2; off >= 1; off >>= 1) {
                u += __shfl_xor_sync(0xffffffffu, u, off);
                wdot += __shfl_xor_sync(0xffffffffu, wdot, off);
            }
            if (valid) {
                const float vi = sh_v[ps * G::RPB + warp * G::RPW + lrow];
                const float c = beta * __fmaf_rn(-alpha, u, vi);
                const float o = __fmaf_rn(c, kappa, alpha * wdot);
                float *dst = Sout + (size_t)i * DK + 4 * lcol;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float4 n;
                    n.x = __fmaf_rn(c, kh[m].x, alpha * s[ps][m].x);
                    n.y = __fmaf_rn(c, kh[m].y, alpha * s[ps][m].y);
                    n.z = __fmaf_rn(c, kh[m].z, alpha * s[ps][m].z);
                    n.w = __fmaf_rn(c, kh[m].w, alpha * s[ps][m].w);
                    st_state(dst + 4 * G::LPR * m, n);
                }
                if (lcol == 0)
                    out[i] = from_f<T>(o);
            }
        }
    } else {
        // padding or bad row: outputs are zeros, no slot is touched
        if (tid < RB) {
            const int i = chunk * RB + tid;
            if (i < p.dv)
                out[i] = from_f<T>(0.f);
        }
    }

    if constexpr (CLUSTER) {
        cluster_wait_acquire(); // every block of the group has read the window
        if (live && writer && tid < DK) {
            const int C = p.channels;
            const int cq = g * DK + tid;
            const int ck = p.hk * DK + g * DK + tid;
            T *wout = reinterpret_cast<T *>(p.conv) + (size_t)ws * (W - 1) * C;
#pragma unroll
            for (int j = 0; j < W - 1; ++j) {
                wout[(size_t)j * C + cq] = from_f<T>(keep_q[j]);
                wout[(size_t)j * C + ck] = from_f<T>(keep_k[j]);
            }
        }
    }
}

// Rows per block: the passes are chosen so that the grid keeps every SM busy
// with several blocks and, in the clustered layer, a qk group fits one
// portable cluster (<= 8 blocks).
template <int DK> int pick_passes(int dv, int group, bool cluster)
{
    using G = Geo<DK>;
    for (int ps : {1, 2, 4}) {
        if (G::RPB * ps > kThreads)
            break;
        const int chunks = (dv + G::RPB * ps - 1) / (G::RPB * ps);
        if (!cluster || group * chunks <= 8)
            return ps;
    }
    return 0;
}

template <typename T, int DK, int PASSES, bool LAYER, int W, bool CLUSTER>
cudaError_t launch_one(const StepArgs &a, cudaStream_t s)
{
    using G = Geo<DK>;
    constexpr int RB = G::RPB * PASSES;
    const int chunks = (a.dv + RB - 1) / RB;
    const long long blocks = (long long)a.rows * a.hv * chunks;
    if (blocks == 0)
        return cudaSuccess;
    auto kern = gdn_state_kernel<T, DK, PASSES, LAYER, W, CLUSTER>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (CLUSTER) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)((a.hv / a.hk) * chunks);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a, chunks);
}

template <typename T, int DK, bool LAYER, int W, bool CLUSTER>
cudaError_t dispatch_passes(const StepArgs &a, cudaStream_t s)
{
    const int ps = pick_passes<DK>(a.dv, a.hv / a.hk, CLUSTER);
    switch (ps) {
    case 1: return launch_one<T, DK, 1, LAYER, W, CLUSTER>(a, s);
    case 2:
        if constexpr (Geo<DK>::RPB * 2 <= kThreads)
            return launch_one<T, DK, 2, LAYER, W, CLUSTER>(a, s);
        break;
    case 4:
        if constexpr (Geo<DK>::RPB * 4 <= kThreads)
            return launch_one<T, DK, 4, LAYER, W, CLUSTER>(a, s);
        break;
    default: break;
    }
    return cudaErrorInvalidConfiguration;
}

template <typename T, bool LAYER, int W, bool CLUSTER>
cudaError_t dispatch_dk(const StepArgs &a, cudaStream_t s)
{
    switch (a.dk) {
    case 16: return dispatch_passes<T, 16, LAYER, W, CLUSTER>(a, s);
    case 32: return dispatch_passes<T, 32, LAYER, W, CLUSTER>(a, s);
    case 64: return dispatch_passes<T, 64, LAYER, W, CLUSTER>(a, s);
    case 128: return dispatch_passes<T, 128, LAYER, W, CLUSTER>(a, s);
    case 256: return dispatch_passes<T, 256, LAYER, W, CLUSTER>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T, int W>
cudaError_t dispatch_layer(const StepArgs &a, cudaStream_t s)
{
    if (a.in_place)
        return dispatch_dk<T, true, W, true>(a, s);
    return dispatch_dk<T, true, W, false>(a, s);
}

} // namespace

bool step_shape_supported(int dk, int dv)
{
    return (dk == 16 || dk == 32 || dk == 64 || dk == 128 || dk == 256) && dv >= 8 && dv <= 512 &&
           dv % 8 == 0;
}

bool layer_shape_supported(int dk, int dv, int group, bool in_place)
{
    if (!step_shape_supported(dk, dv) || group < 1)
        return false;
    if (!in_place)
        return true;
    switch (dk) {
    case 16: return pick_passes<16>(dv, group, true) > 0;
    case 32: return pick_passes<32>(dv, group, true) > 0;
    case 64: return pick_passes<64>(dv, group, true) > 0;
    case 128: return pick_passes<128>(dv, group, true) > 0;
    case 256: return pick_passes<256>(dv, group, true) > 0;
    default: return false;
    }
}

cudaError_t launch_gdn_step(const StepArgs &a, int dtype, cudaStream_t s)
{
    if (dtype == GDN_BF16)
        return dispatch_dk<__nv_bfloat16, false, 2, false>(a, s);
    return dispatch_dk<float, false, 2, false>(a, s);
}

cudaError_t launch_gdn_layer(const StepArgs &a, int dtype, cudaStream_t s)
{
    switch (a.width) {
    case 2: return dtype == GDN_BF16 ? dispatch_layer<__nv_bfloat16, 2>(a, s) : dispatch_layer<float, 2>(a, s);
    case 3: return dtype == GDN_BF16 ? dispatch_layer<__nv_bfloat16, 3>(a, s) : dispatch_layer<float, 3>(a, s);
    case 4: return dtype == GDN_BF16 ? dispatch_layer<__nv_bfloat16, 4>(a, s) : dispatch_layer<float, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gdn
