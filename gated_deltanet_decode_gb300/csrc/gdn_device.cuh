// Device-side helpers shared by the GDN decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// ---------------------------------------------------------------------------
// Activation types: fp32 or bf16, converted to fp32 for all arithmetic.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// Round an fp32 value to the activation type and back (the value a separate
// kernel would have stored and the next one would have read).
template <typename T> __device__ __forceinline__ float round_act(float x)
{
    return to_f(from_f<T>(x));
}

// ---------------------------------------------------------------------------
// State stream: 16-byte loads that skip L1 (each byte is touched once), and
// plain 16-byte stores.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 ld_state(const float *p)
{
    float4 v;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_state(float *p, float4 v)
{
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Gates (fp32, with CUDA's expf / log1pf).
//   alpha = exp(-exp(A_log) * softplus(a + dt_bias)),  softplus(x) = x above 20
//   beta  = 1 / (1 + exp(-b))
// ---------------------------------------------------------------------------
__device__ __forceinline__ float softplus_f(float x)
{
    return x > 20.0f ? x : log1pf(expf(x));
}
__device__ __forceinline__ float gate_alpha(float A_log, float a, float dt_bias)
{
    float rate = expf(A_log);
    float g = rate == 0.0f ? 0.0f : rate * softplus_f(a + dt_bias);
    return expf(-g);
}
__device__ __forceinline__ float gate_beta(float b)
{
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-b)));
}

// ---------------------------------------------------------------------------
// Depthwise causal conv of one channel for one token.  win[j] are the
// previous W-1 inputs (oldest first); tap W-1 multiplies x.  The same routine
// serves the standalone conv and the fused layer, so both round identically.
// ---------------------------------------------------------------------------
template <int W>
__device__ __forceinline__ float conv_channel(const float (&win)[W - 1], float x, const float (&w)[W],
                                              float bias, bool silu)
{
    float pre = bias;
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
        pre = __fmaf_rn(w[j], win[j], pre);
    pre = __fmaf_rn(w[W - 1], x, pre);
    if (silu)
        pre = __fdiv_rn(pre, __fadd_rn(1.0f, expf(-pre)));
    return pre;
}

// Programmatic dependent launch: kernels are launched with the PDL attribute,
// so a kernel's CTAs may be scheduled while the previous kernel on the stream
// drains.  Every kernel calls this before its first global-memory access; it
// returns once the previous grid has completed and its writes are visible
// (at once when there is no such dependency), so stream order is preserved.
__device__ __forceinline__ void wait_prior_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kern` on `s` with the programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Sticky device error word: the first error code wins.
__device__ __forceinline__ void report(int *err, int code)
{
    if (err)
        atomicCAS(err, 0, code);
}

// Row classification shared by every slot-indexed kernel.
//   0 = padding (read slot 0), 1 = real, -1 = bad (reported by the caller).
// Padding rows address only the null slot and leave it untouched ("mstar PR
// #965" and "mstar PR #1127", "What changed").  A twin step writes the
// request's other slot ("mstar PR #1139", "What changed"), so a twin write
// slot equal to the read slot is bad.
__device__ __forceinline__ int classify_row(int rs, int ws, int num_slots, bool in_place)
{
    if (rs == 0)
        return 0;
    if (rs < 0 || rs >= num_slots)
        return -1;
    if (in_place)
        return 1;
    if (ws <= 0 || ws >= num_slots || ws == rs)
        return -1;
    return 1;
}

// Sequence classification of the many-token kernels (0 padding, 1 real,
// -1 bad): a token range outside [0, total_tokens) is bad; with token slots
// every token's slot must be a real slot other than the read slot; otherwise
// as classify_row.
__device__ __forceinline__ int classify_seq(int rs, int ws, bool in_place, const int32_t *token_slot,
                                            int t0, int t1, int total_tokens, int num_slots)
{
    if (t0 < 0 || t1 < t0 || t1 > total_tokens)
        return -1;
    if (token_slot) {
        const int cls = classify_row(rs, rs, num_slots, true);
        if (cls != 1)
            return cls;
        for (int t = t0; t < t1; ++t) {
            const int s = token_slot[t];
            if (s <= 0 || s >= num_slots || s == rs)
                return -1;
        }
        return 1;
    }
    return classify_row(rs, ws, num_slots, in_place);
}

} // namespace gdn
