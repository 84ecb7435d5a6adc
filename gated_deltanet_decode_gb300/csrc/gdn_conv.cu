// causal_conv1d_decode: depthwise causal conv for one token a row over a
// slot-indexed conv window pool, sm_103a ("mstar PR #1139", section "What
// changed": the conv state update for one token a row, with a write slot).
//
// A thread owns 8 consecutive channels of one row: it reads the W-1 window
// entries of its channels (16 bytes each in bf16), the token, the W taps and
// the bias, writes the output and the shifted window.  In place (no write
// slot) the thread reads its window before overwriting it, and no other
// thread touches those channels, so no synchronisation is needed.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8; // channels per thread

// Eight activations as loaded (for rows kept in registers before use).
template <typename T> struct Raw8;
template <> struct Raw8<float> { float4 a, b; };
template <> struct Raw8<__nv_bfloat16> { uint4 u; };

template <typename T> struct Vec8;
template <> struct Vec8<float> {
    static __device__ __forceinline__ Raw8<float> ldraw(const float *p)
    {
        return {*reinterpret_cast<const float4 *>(p), *reinterpret_cast<const float4 *>(p + 4)};
    }
    static __device__ __forceinline__ Raw8<float> zero()
    {
        return {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    }
    static __device__ __forceinline__ void unpack(const Raw8<float> &r, float (&v)[8])
    {
        v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
        v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
    }
    static __device__ __forceinline__ void straw(float *p, const Raw8<float> &r)
    {
        *reinterpret_cast<float4 *>(p) = r.a;
        *reinterpret_cast<float4 *>(p + 4) = r.b;
    }
    static __device__ __forceinline__ void load(const float *p, float (&v)[8])
    {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        const float4 b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    static __device__ __forceinline__ void store(float *p, const float (&v)[8])
    {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
};
template <> struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ Raw8<__nv_bfloat16> ldraw(const __nv_bfloat16 *p)
    {
        return {*reinterpret_cast<const uint4 *>(p)};
    }
    static __device__ __forceinline__ Raw8<__nv_bfloat16> zero() { return {make_uint4(0u, 0u, 0u, 0u)}; }
    static __device__ __forceinline__ void unpack(const Raw8<__nv_bfloat16> &r, float (&v)[8])
    {
        const uint32_t w[4] = {r.u.x, r.u.y, r.u.z, r.u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void straw(__nv_bfloat16 *p, const Raw8<__nv_bfloat16> &r)
    {
        *reinterpret_cast<uint4 *>(p) = r.u;
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&v)[8])
    {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&v)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// The same for four activations (the conv over a sequence: fewer registers a
// thread, so more threads an SM hide its latencies).
template <typename T> struct Raw4v;
template <> struct Raw4v<float> { float4 a; };
template <> struct Raw4v<__nv_bfloat16> { uint2 u; };

template <typename T> struct Vec4v;
template <> struct Vec4v<float> {
    static __device__ __forceinline__ Raw4v<float> ldraw(const float *p) { return {*reinterpret_cast<const float4 *>(p)}; }
    static __device__ __forceinline__ Raw4v<float> zero() { return {make_float4(0.f, 0.f, 0.f, 0.f)}; }
    static __device__ __forceinline__ void unpack(const Raw4v<float> &r, float (&v)[4])
    {
        v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
    }
    static __device__ __forceinline__ void straw(float *p, const Raw4v<float> &r)
    {
        *reinterpret_cast<float4 *>(p) = r.a;
    }
    static __device__ __forceinline__ void load(const float *p, float (&v)[4])
    {
        unpack(ldraw(p), v);
    }
    static __device__ __forceinline__ void store(float *p, const float (&v)[4])
    {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec4v<__nv_bfloat16> {
    static __device__ __forceinline__ Raw4v<__nv_bfloat16> ldraw(const __nv_bfloat16 *p)
    {
        return {*reinterpret_cast<const uint2 *>(p)};
    }
    static __device__ __forceinline__ Raw4v<__nv_bfloat16> zero() { return {make_uint2(0u, 0u)}; }
    static __device__ __forceinline__ void unpack(const Raw4v<__nv_bfloat16> &r, float (&v)[4])
    {
        const uint32_t w[2] = {r.u.x, r.u.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void straw(__nv_bfloat16 *p, const Raw4v<__nv_bfloat16> &r)
    {
        *reinterpret_cast<uint2 *>(p) = r.u;
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&v)[4])
    {
        unpack(ldraw(p), v);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&v)[4])
    {
        uint32_t w[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
    }
};

// the helpers of NV activations a thread
template <typename T, int NV> struct VecOf;
template <typename T> struct VecOf<T, 8> {
    using V = Vec8<T>;
    using R = Raw8<T>;
};
template <typename T> struct VecOf<T, 4> {
    using V = Vec4v<T>;
    using R = Raw4v<T>;
};

template <typename T, int W>
__global__ void __launch_bounds__(kThreads) conv_decode_kernel(const ConvArgs p, int groups_per_row)
{
    wait_prior_grid();
    const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
    const int r = (int)(gid / groups_per_row);
    const int c0 = (int)(gid % groups_per_row) * kVec;
    if (r >= p.rows)
        return;
    const int C = p.channels;
    const int rs = p.read_slot[r];
    const bool in_place = p.write_slot == nullptr;
    const int ws = in_place ? rs : p.write_slot[r];
    const int cls = classify_row(rs, ws, p.num_slots, in_place);
    T *out = reinterpret_cast<T *>(p.out) + (size_t)r * C + c0;
    if (cls != 1) {
        if (cls < 0 && c0 == 0)
            report(p.err, GDN_DEVERR_BAD_SLOT);
        float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        Vec8<T>::store(out, z);
        return;
    }
    const T *conv_in = reinterpret_cast<const T *>(p.conv) + (size_t)rs * (W - 1) * C + c0;
    T *conv_out = reinterpret_cast<T *>(p.conv) + (size_t)ws * (W - 1) * C + c0;

    float win[W - 1][8];
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
        Vec8<T>::load(conv_in + (size_t)j * C, win[j]);
    float x[8];
    Vec8<T>::load(reinterpret_cast<const T *>(p.x) + (size_t)r * p.x_stride + c0, x);
    // taps of channels c0..c0+7 are 8*W consecutive values: channel i, tap j at i*W + j
    float taps[8 * W];
    {
        const T *wp = reinterpret_cast<const T *>(p.w) + (size_t)c0 * W;
#pragma unroll
        for (int t = 0; t < W; ++t) {
            float tmp[8];
            Vec8<T>::load(wp + 8 * t, tmp);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                taps[8 * t + i] = tmp[i];
        }
    }
    float bias[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (p.bias)
        Vec8<T>::load(reinterpret_cast<const T *>(p.bias) + c0, bias);

    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float wi[W], wn[W - 1];
#pragma unroll
        for (int j = 0; j < W; ++j)
            wi[j] = taps[i * W + j];
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
            wn[j] = win[j][i];
        y[i] = conv_channel<W>(wn, x[i], wi, bias[i], p.silu != 0);
    }
    Vec8<T>::store(out, y);
#pragma unroll
    for (int j = 0; j + 1 < W - 1; ++j)
        Vec8<T>::store(conv_out + (size_t)j * C, win[j + 1]);
    Vec8<T>::store(conv_out + (size_t)(W - 2) * C, x);
}

// The conv over many tokens a sequence ("mstar PR #1139", section "Why":
// prefill keeps the state in place).  A token's output depends only on it and
// the W-1 inputs before it, so the tokens run in parallel: a token thread
// (one per run of kRun tokens and NV = 4 channels) takes the run's tokens that
// are at least W-1 into their sequence; it loads every input row they need
// (the run's and the W-1 before it) at once, so many loads are in flight,
// and reads only the packed inputs; a window thread (one per
// sequence and NV channels) takes the first W-1 tokens, which read the stored
// window, and then writes the new window -- reads before writes in one
// thread, so in place is safe.  Each output equals one causal_conv1d_decode
// call.  With token slots, the window after each token goes to that token's
// slot (the window thread writes those of the first W-1 tokens).
template <typename T, int W, int NV>
__device__ __forceinline__ void convN(const float (&win)[W - 1][NV], const float (&x)[NV], const float *taps,
                                      const float (&bias)[NV], bool silu, float (&y)[NV])
{
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        float wi[W], wn[W - 1];
#pragma unroll
        for (int j = 0; j < W; ++j)
            wi[j] = taps[i * W + j];
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
            wn[j] = win[j][i];
        y[i] = conv_channel<W>(wn, x[i], wi, bias[i], silu);
    }
}

constexpr int kRun = 4; // tokens a token thread walks

// The sequence holding token `tok`: the last r with cu_seqlens[r] <= tok.
__device__ __forceinline__ int seq_of(const int32_t *cu, int nseq, long long tok)
{
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= tok)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// the taps (channel-major, W a channel) and bias of channels c0 .. c0 + NV - 1
template <typename T, int W, int NV>
__device__ __forceinline__ void load_taps(const ConvPrefillArgs &p, int c0, float (&taps)[NV * W], float (&bias)[NV])
{
    using VV = typename VecOf<T, NV>::V;
    const T *wp = reinterpret_cast<const T *>(p.w) + (size_t)c0 * W;
#pragma unroll
    for (int t = 0; t < W; ++t) {
        float tmp[NV];
        VV::load(wp + NV * t, tmp);
#pragma unroll
        for (int i = 0; i < NV; ++i)
            taps[NV * t + i] = tmp[i];
    }
#pragma unroll
    for (int i = 0; i < NV; ++i)
        bias[i] = 0.f;
    if (p.bias)
        VV::load(reinterpret_cast<const T *>(p.bias) + c0, bias);
}

template <typename T, int W, int NV>
__global__ void __launch_bounds__(kThreads, 3) conv_prefill_kernel(const ConvPrefillArgs p, int groups_per_row)
{
    using VV = typename VecOf<T, NV>::V;
    wait_prior_grid();
    const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
    const long long n_window = (long long)p.nseq * groups_per_row;
    const int C = p.channels;
    T *conv = reinterpret_cast<T *>(p.conv);
    const T *xs = reinterpret_cast<const T *>(p.x);
    const bool in_place = p.write_slot == nullptr || p.token_slot != nullptr;
    const bool silu = p.silu != 0;
    T *out = nullptr;
    float taps[NV * W], bias[NV];
    float win[W - 1][NV], x[NV], y[NV];

    if (gid >= n_window) {
        // ------------------------- token thread -------------------------
        const long long g2 = gid - n_window;
        const long long run = g2 / groups_per_row;
        const int c0 = (int)(g2 % groups_per_row) * NV;
        const long long first = run * kRun;
        if (first >= p.total_tokens)
            return;
        const long long last = first + kRun < p.total_tokens ? first + kRun : p.total_tokens;
        out = reinterpret_cast<T *>(p.out) + c0;
        load_taps<T, W, NV>(p, c0, taps, bias);
        // every input row the run needs (its tokens and the W-1 before them),
        // all loads in flight before any is used; rows outside [0, T) read as zeros
        constexpr int NR = kRun + W - 1;
        typename VecOf<T, NV>::R raw[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const long long tok = first - (W - 1) + i;
            raw[i] = tok >= 0 && tok < p.total_tokens ? VV::ldraw(xs + (size_t)tok * C + c0) : VV::zero();
        }
        int r = -1, t0 = 0, t1 = 0, cls = 0;
#pragma unroll
        for (int i = 0; i < kRun; ++i) {
            const long long tok = first + i;
            if (tok >= last)
                break;
            if (r < 0 || tok >= t1) {
                r = seq_of(p.cu_seqlens, p.nseq, tok);
                t0 = p.cu_seqlens[r];
                t1 = p.cu_seqlens[r + 1];
                const int rs = p.read_slot[r];
                const int ws = in_place ? rs : p.write_slot[r];
                cls = classify_seq(rs, ws, in_place, p.token_slot, t0, t1, p.total_tokens, p.num_slots);
            }
            if (tok < t0 || tok >= t1 || tok - t0 < W - 1)
                continue; // not in this sequence's range, or a window thread's token
            if (cls != 1) {
                float z[NV];
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    z[i] = 0.f;
                VV::store(out + (size_t)tok * C, z);
                continue;
            }
            // the W-1 inputs before tok are rows i..i+W-2 (all in this sequence)
#pragma unroll
            for (int j = 0; j < W - 1; ++j)
                VV::unpack(raw[i + j], win[j]);
            VV::unpack(raw[i + W - 1], x);
            convN<T, W, NV>(win, x, taps, bias, silu, y);
            VV::store(out + (size_t)tok * C, y);
            if (p.token_slot) {
                // the window after tok: rows i+1..i+W-1, as they were read
                const int ts = p.token_slot[tok];
#pragma unroll
                for (int j = 0; j < W - 1; ++j)
                    VV::straw(conv + ((size_t)ts * (W - 1) + j) * C + c0, raw[i + 1 + j]);
            }
        }
        return;
    }

    // ------------------------- window thread --------------------------
    const int r = (int)(gid / groups_per_row);
    const int c0 = (int)(gid % groups_per_row) * NV;
    const int t0 = p.cu_seqlens[r], t1 = p.cu_seqlens[r + 1];
    const int rs = p.read_slot[r];
    const int ws = in_place ? rs : p.write_slot[r];
    const int cls = classify_seq(rs, ws, in_place, p.token_slot, t0, t1, p.total_tokens, p.num_slots);
    out = reinterpret_cast<T *>(p.out) + c0;
    if (cls != 1) {
        float z[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i)
            z[i] = 0.f;
        if (cls < 0 && c0 == 0)
            report(p.err, GDN_DEVERR_BAD_SLOT);
        if (t0 >= 0 && t1 >= t0 && t1 <= p.total_tokens)
            for (int t = t0; t < t1 && t < t0 + W - 1; ++t)
                VV::store(out + (size_t)t * C, z);
        return;
    }
    load_taps<T, W, NV>(p, c0, taps, bias);
    // the first W-1 tokens, then the new window
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
        VV::load(conv + ((size_t)rs * (W - 1) + j) * C + c0, win[j]);
    const int n = t1 - t0;
    const int head = n < W - 1 ? n : W - 1;
    for (int t = t0; t < t0 + head; ++t) {
        VV::load(xs + (size_t)t * C + c0, x);
        convN<T, W, NV>(win, x, taps, bias, silu, y);
        VV::store(out + (size_t)t * C, y);
        // the window moves on by one token; values stay in the activation type
#pragma unroll
        for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                win[j][i] = win[j + 1][i];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            win[W - 2][i] = x[i];
        if (p.token_slot) {
            const int ts = p.token_slot[t];
#pragma unroll
            for (int j = 0; j < W - 1; ++j)
                VV::store(conv + ((size_t)ts * (W - 1) + j) * C + c0, win[j]);
        }
    }
    if (!p.token_slot) {
        // the window after the last token: the last W-1 inputs (with the old
        // window's tail when the sequence is shorter than that)
        if (n > W - 1) {
#pragma unroll
            for (int j = 0; j < W - 1; ++j)
                VV::load(xs + (size_t)(t1 - (W - 1) + j) * C + c0, win[j]);
        }
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
            VV::store(conv + ((size_t)ws * (W - 1) + j) * C + c0, win[j]);
    }
}

// channels a thread of the conv over a sequence (fewer registers than 8: more
// threads an SM to hide the exact SiLU's latency)
constexpr int kVecPrefill = 4;

template <typename T, int W>
cudaError_t launch_prefill_w(const ConvPrefillArgs &a, cudaStream_t s)
{
    const int groups = a.channels / kVecPrefill;
    const long long runs = ((long long)a.total_tokens + kRun - 1) / kRun;
    const long long threads = ((long long)a.nseq + runs) * groups;
    if (a.nseq == 0 || threads == 0)
        return cudaSuccess;
    const long long blocks = (threads + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffll)
        return cudaErrorInvalidValue;
    return launch_pdl(conv_prefill_kernel<T, W, kVecPrefill>, dim3((unsigned)blocks), dim3(kThreads), 0, s, a,
                      groups);
}

template <typename T>
cudaError_t launch_prefill_t(const ConvPrefillArgs &a, cudaStream_t s)
{
    switch (a.width) {
    case 2: return launch_prefill_w<T, 2>(a, s);
    case 3: return launch_prefill_w<T, 3>(a, s);
    case 4: return launch_prefill_w<T, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T, int W>
cudaError_t launch_w(const ConvArgs &a, cudaStream_t s)
{
    const int groups = a.channels / kVec;
    const long long threads = (long long)a.rows * groups;
    if (threads == 0)
        return cudaSuccess;
    const long long blocks = (threads + kThreads - 1) / kThreads;
    return launch_pdl(conv_decode_kernel<T, W>, dim3((unsigned)blocks), dim3(kThreads), 0, s, a, groups);
}

template <typename T>
cudaError_t launch_t(const ConvArgs &a, cudaStream_t s)
{
    switch (a.width) {
    case 2: return launch_w<T, 2>(a, s);
    case 3: return launch_w<T, 3>(a, s);
    case 4: return launch_w<T, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

cudaError_t launch_conv(const ConvArgs &a, int dtype, cudaStream_t s)
{
    return dtype == GDN_BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

cudaError_t launch_conv_prefill(const ConvPrefillArgs &a, int dtype, cudaStream_t s)
{
    return dtype == GDN_BF16 ? launch_prefill_t<__nv_bfloat16>(a, s) : launch_prefill_t<float>(a, s);
}

} // namespace gdn
