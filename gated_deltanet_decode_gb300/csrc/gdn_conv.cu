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

template <typename T> struct Vec8;
template <> struct Vec8<float> {
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
// prefill keeps the state in place): a thread owns 8 channels of one
// sequence, keeps their window in registers and walks the tokens in order,
// so each token's output equals one causal_conv1d_decode call.  The window
// after the last token goes to the write slot (or back in place); with token
// slots, the window after every token goes to that token's slot.
template <typename T, int W>
__global__ void __launch_bounds__(kThreads) conv_prefill_kernel(const ConvPrefillArgs p, int groups_per_row)
{
    wait_prior_grid();
    const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
    const int r = (int)(gid / groups_per_row);
    const int c0 = (int)(gid % groups_per_row) * kVec;
    if (r >= p.nseq)
        return;
    const int C = p.channels;
    const int t0 = p.cu_seqlens[r], t1 = p.cu_seqlens[r + 1];
    const int rs = p.read_slot[r];
    const bool in_place = p.write_slot == nullptr || p.token_slot != nullptr;
    const int ws = in_place ? rs : p.write_slot[r];
    const int cls = classify_seq(rs, ws, in_place, p.token_slot, t0, t1, p.total_tokens, p.num_slots);
    T *out = reinterpret_cast<T *>(p.out) + c0;
    if (cls != 1) {
        if (cls < 0 && c0 == 0)
            report(p.err, GDN_DEVERR_BAD_SLOT);
        if (t0 >= 0 && t1 >= t0 && t1 <= p.total_tokens) {
            float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int t = t0; t < t1; ++t)
                Vec8<T>::store(out + (size_t)t * C, z);
        }
        return;
    }
    T *conv = reinterpret_cast<T *>(p.conv);
    float win[W - 1][8];
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
        Vec8<T>::load(conv + ((size_t)rs * (W - 1) + j) * C + c0, win[j]);
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
    const T *xp = reinterpret_cast<const T *>(p.x) + c0;
    for (int t = t0; t < t1; ++t) {
        float x[8], y[8];
        Vec8<T>::load(xp + (size_t)t * C, x);
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
        Vec8<T>::store(out + (size_t)t * C, y);
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
                Vec8<T>::store(conv + ((size_t)ts * (W - 1) + j) * C + c0, win[j]);
        }
    }
    if (!p.token_slot) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
            Vec8<T>::store(conv + ((size_t)ws * (W - 1) + j) * C + c0, win[j]);
    }
}

template <typename T, int W>
cudaError_t launch_prefill_w(const ConvPrefillArgs &a, cudaStream_t s)
{
    const int groups = a.channels / kVec;
    const long long threads = (long long)a.nseq * groups;
    if (threads == 0)
        return cudaSuccess;
    const long long blocks = (threads + kThreads - 1) / kThreads;
    return launch_pdl(conv_prefill_kernel<T, W>, dim3((unsigned)blocks), dim3(kThreads), 0, s, a, groups);
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
