// Device code shared by the two chunked-prefill kernels (sm_103a): the chunk
// geometry, bf16 head/tail splits, mma.sync fragments, activation loads, and
// the blocked inverse of the chunk's unit lower-triangular matrix.  Included
// by one translation unit each; everything here has internal linkage.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_device.cuh"

namespace gdn {
namespace {

typedef __nv_bfloat16 bf16;

constexpr int CK = 64;      // tokens a chunk
constexpr int CD = 128;     // dk = dv
// Row stride (fp32) of the fp32 [token][token] work tiles: 288-byte rows, so
// the 8-byte (row g, columns 2c, 2c+1) accesses of an mma fragment put each
// half-warp's four rows on distinct groups of eight banks.
constexpr int LDF = CK + 8;

// ---------------------------------------------------------------------------
// Tensor-core helpers (mma.sync m16n8k16, bf16 in, fp32 accumulate).
// Fragment layout, g = lane / 4, c = lane % 4:
//   A 16x16: a0 = (g, 2c..2c+1), a1 = (g+8, 2c..), a2 = (g, 2c+8..), a3 = (g+8, 2c+8..)
//   B 16x8:  b0 = (k 2c..2c+1, n g), b1 = (k 2c+8..2c+9, n g)
//   D 16x8:  d0 = (g, 2c), d1 = (g, 2c+1), d2 = (g+8, 2c), d3 = (g+8, 2c+1)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t *>(&v); }

// Split (x, y) into bf16 heads and tails: x = hi.x + lo.x to 2^-17 relative.
__device__ __forceinline__ void split2(float x, float y, uint32_t &hi, uint32_t &lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    hi = bits(h);
    lo = bits(__floats2bfloat162_rn(x - hf.x, y - hf.y));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d += (ah + al)(bh + bl), dropping al*bl (about 2^-34 relative).
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], uint32_t bh0,
                                     uint32_t bh1, uint32_t bl0, uint32_t bl1)
{
    mma16816(d, al[0], al[1], al[2], al[3], bh0, bh1);
    mma16816(d, ah[0], ah[1], ah[2], ah[3], bl0, bl1);
    mma16816(d, ah[0], ah[1], ah[2], ah[3], bh0, bh1);
}

// A fragment of rows m0.., columns k0.. of a row-major bf16 tile X (row stride ld).
__device__ __forceinline__ void lda(uint32_t (&a)[4], const bf16 *X, int ld, int m0, int k0, int g, int c)
{
    const bf16 *p = X + (m0 + g) * ld + k0 + 2 * c;
    a[0] = *reinterpret_cast<const uint32_t *>(p);
    a[1] = *reinterpret_cast<const uint32_t *>(p + 8 * ld);
    a[2] = *reinterpret_cast<const uint32_t *>(p + 8);
    a[3] = *reinterpret_cast<const uint32_t *>(p + 8 * ld + 8);
}

// B fragment with B[k][n] = X[n][k]: columns n0.., rows k0.. (X row-major, stride ld).
__device__ __forceinline__ void ldb(uint32_t &b0, uint32_t &b1, const bf16 *X, int ld, int n0, int k0, int g, int c)
{
    const bf16 *p = X + (n0 + g) * ld + k0 + 2 * c;
    b0 = *reinterpret_cast<const uint32_t *>(p);
    b1 = *reinterpret_cast<const uint32_t *>(p + 8);
}

// B fragments of two adjacent 8-column tiles with B[k][n] = X[k][n] (X
// row-major [k][n], stride ld): rows k0..k0+15, columns n0..n0+15.  One
// transposing ldmatrix; lane l names row l%8 of 8x8 matrix l/8, matrix m
// covering rows k0 + 8(m&1), columns n0 + 8(m>>1).
__device__ __forceinline__ void ldb_trans2(uint32_t (&b)[4], const bf16 *X, int ld, int k0, int n0, int lane)
{
    const int m = lane >> 3, r = lane & 7;
    const bf16 *p = X + (k0 + 8 * (m & 1) + r) * ld + n0 + 8 * (m >> 1);
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
                 : "r"(a));
}

// Split accumulator tiles c0 (columns 0..7) and c1 (8..15) of one 16x16
// block into the A fragments of that block (rows the same, k = columns).
__device__ __forceinline__ void acc_to_a(uint32_t (&ah)[4], uint32_t (&al)[4], const float (&c0)[4],
                                         const float (&c1)[4])
{
    split2(c0[0], c0[1], ah[0], al[0]);
    split2(c0[2], c0[3], ah[1], al[1]);
    split2(c1[0], c1[1], ah[2], al[2]);
    split2(c1[2], c1[3], ah[3], al[3]);
}

// A fragment of a row-major fp32 tile (rows m0.., columns k0..), split.
__device__ __forceinline__ void lda_f32(uint32_t (&ah)[4], uint32_t (&al)[4], const float *X, int ld, int m0, int k0,
                                        int g, int c)
{
    const float *p = X + (m0 + g) * ld + k0 + 2 * c; // 8-byte aligned: ld and k0 even
    float2 v = *reinterpret_cast<const float2 *>(p);
    split2(v.x, v.y, ah[0], al[0]);
    v = *reinterpret_cast<const float2 *>(p + 8 * ld);
    split2(v.x, v.y, ah[1], al[1]);
    v = *reinterpret_cast<const float2 *>(p + 8);
    split2(v.x, v.y, ah[2], al[2]);
    v = *reinterpret_cast<const float2 *>(p + 8 * ld + 8);
    split2(v.x, v.y, ah[3], al[3]);
}

// B fragment with B[k][n] = X[k][n] of a row-major fp32 tile (rows k0..,
// columns n0..), split.
__device__ __forceinline__ void ldb_f32(uint32_t &bh0, uint32_t &bh1, uint32_t &bl0, uint32_t &bl1, const float *X,
                                        int ld, int k0, int n0, int g, int c)
{
    const float *p = X + (k0 + 2 * c) * ld + n0 + g;
    split2(p[0], p[ld], bh0, bl0);
    split2(p[8 * ld], p[9 * ld], bh1, bl1);
}

// Four activations as loaded (one 16- or 8-byte load), then as fp32.
template <typename T> struct Raw4;
template <> struct Raw4<float> { float4 v; };
template <> struct Raw4<bf16> { uint2 v; };
template <typename T> __device__ __forceinline__ Raw4<T> ldraw(const T *p);
template <> __device__ __forceinline__ Raw4<float> ldraw<float>(const float *p)
{
    return {*reinterpret_cast<const float4 *>(p)};
}
template <> __device__ __forceinline__ Raw4<bf16> ldraw<bf16>(const bf16 *p)
{
    return {*reinterpret_cast<const uint2 *>(p)};
}
template <typename T> __device__ __forceinline__ Raw4<T> raw_zero();
template <> __device__ __forceinline__ Raw4<float> raw_zero<float>() { return {make_float4(0.f, 0.f, 0.f, 0.f)}; }
template <> __device__ __forceinline__ Raw4<bf16> raw_zero<bf16>() { return {make_uint2(0u, 0u)}; }
__device__ __forceinline__ void unpack(float (&v)[4], const Raw4<float> &r)
{
    v[0] = r.v.x, v[1] = r.v.y, v[2] = r.v.z, v[3] = r.v.w;
}
__device__ __forceinline__ void unpack(float (&v)[4], const Raw4<bf16> &r)
{
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.v.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.v.y));
    v[0] = a.x, v[1] = a.y, v[2] = b.x, v[3] = b.y;
}

// 16-byte asynchronous copy global -> shared; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <typename T> __device__ __forceinline__ void store2(T *p, float x, float y);
template <> __device__ __forceinline__ void store2<float>(float *p, float x, float y)
{
    *reinterpret_cast<float2 *>(p) = make_float2(x, y);
}
template <> __device__ __forceinline__ void store2<bf16>(bf16 *p, float x, float y)
{
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x, y);
}

constexpr float kEps = 1e-6f; // L2-norm epsilon, as in the decode kernels

// ---------------------------------------------------------------------------
// A chunk's gates, by one warp (tokens lane and lane + 32 of the nn live
// ones; zero past them): into G = [running sum of log alpha | beta | e^G |
// e^{G_C - G}] x CK, with alpha = exp(-rate softplus(a + dt_bias)) taken in
// log form and beta = sigmoid(b).
// ---------------------------------------------------------------------------
template <typename TA>
__device__ __forceinline__ void chunk_gates(float *G, const TA (&ra)[2], const TA (&rb)[2], int nn, float rate,
                                            float dtb, int lane)
{
    float la[2], bt[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int tt = lane + 32 * i;
        la[i] = 0.f, bt[i] = 0.f;
        if (tt < nn) {
            la[i] = rate == 0.f ? 0.f : -rate * softplus_f(to_f(ra[i]) + dtb);
            bt[i] = gate_beta(to_f(rb[i]));
        }
    }
    float s0 = la[0], s1 = la[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float x0 = __shfl_up_sync(0xffffffffu, s0, o);
        const float x1 = __shfl_up_sync(0xffffffffu, s1, o);
        if (lane >= o)
            s0 += x0, s1 += x1;
    }
    s1 += __shfl_sync(0xffffffffu, s0, 31);
    const float gc = __shfl_sync(0xffffffffu, s1, 31);
    G[lane] = s0, G[lane + 32] = s1;
    G[CK + lane] = bt[0], G[CK + lane + 32] = bt[1];
    G[2 * CK + lane] = expf(s0), G[2 * CK + lane + 32] = expf(s1);
    G[3 * CK + lane] = expf(gc - s0), G[3 * CK + lane + 32] = expf(gc - s1);
}

// ---------------------------------------------------------------------------
// T = (I + A)^{-1} for the chunk's strictly lower A (fp32 [CK][LDF] in AF):
// the 16x16 diagonal blocks by forward substitution on unit vectors, one
// column a thread (threads 0..CK-1), into XF.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void t_diagonal(const float *AF, float *XF, int tid)
{
    const int base = 16 * (tid >> 4), col = tid & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float *arow = AF + (base + r) * LDF + base;
        float acc = r == col ? 1.f : 0.f;
#pragma unroll
        for (int s = 0; s < r; ++s)
            acc = fmaf(-arow[s], x[s], acc);
        x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r)
        XF[(base + r) * LDF + base + col] = x[r];
}

// The blocks below the diagonal, by distance d from it, one warp a block
// (J = warp): X = sum_{K=J}^{I-1} A_IK T_KJ, parked in A's unused block
// (J, I); T_IJ = -T_II X.  Every thread of the CTA calls it (it holds the
// CTA barriers between distances).
__device__ __forceinline__ void t_below_diagonal(float *AF, float *XF, int warp, int g, int c)
{
#pragma unroll 1
    for (int d = 1; d < CK / 16; ++d) {
        const int J = warp, I = warp + d;
        if (I < CK / 16) {
            float x[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int K = J; K < I; ++K) {
                uint32_t ah[4], al[4];
                lda_f32(ah, al, AF, LDF, 16 * I, 16 * K, g, c);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    uint32_t bh0, bh1, bl0, bl1;
                    ldb_f32(bh0, bh1, bl0, bl1, XF, LDF, 16 * K, 16 * J + 8 * nt, g, c);
                    mma3(x[nt], ah, al, bh0, bh1, bl0, bl1);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<float2 *>(AF + (16 * J + g + 8 * hr) * LDF + 16 * I + 8 * nt + 2 * c) =
                        make_float2(x[nt][2 * hr], x[nt][2 * hr + 1]);
            __syncwarp();
            float tij[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            uint32_t ah[4], al[4];
            lda_f32(ah, al, XF, LDF, 16 * I, 16 * I, g, c);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t bh0, bh1, bl0, bl1;
                ldb_f32(bh0, bh1, bl0, bl1, AF, LDF, 16 * J, 16 * I + 8 * nt, g, c);
                mma3(tij[nt], ah, al, bh0, bh1, bl0, bl1);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<float2 *>(XF + (16 * I + g + 8 * hr) * LDF + 16 * J + 8 * nt + 2 * c) =
                        make_float2(-tij[nt][2 * hr], -tij[nt][2 * hr + 1]);
        }
        __syncthreads();
    }
}

} // namespace
} // namespace gdn
