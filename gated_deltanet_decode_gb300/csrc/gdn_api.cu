// C ABI of the GDN decode library: argument checks, pools, the sticky device
// error word, and the small kernels (commit, slot zeroing, traffic probes).
// The heavy kernels live in gdn_stream.cu and gdn_conv.cu.  The pools follow
// "mstar PR #1139", "What changed" (a request holds two state slots; a decode
// step reads one and writes the other; commit swaps them; release and
// rollback zero both, "Tests") and "mstar PR #1127", "What changed" (padding
// rows sit on slot 0, which stays zero).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_ptx.cuh"

#define GDN_ABI_VERSION 1

// ---------------------------------------------------------------------------
// error reporting
// ---------------------------------------------------------------------------
namespace {

thread_local char t_msg[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof t_msg, fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    t_msg[0] = '\0';
    return GDN_OK;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(GDN_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dtype_ok(int dtype) { return dtype == GDN_F32 || dtype == GDN_BF16; }

size_t dtype_size(int dtype) { return dtype == GDN_BF16 ? 2 : 4; }

} // namespace

// ---------------------------------------------------------------------------
// The device error word.  One int per device, in the library's own module
// memory.  Host code cannot use the symbol as a pointer; its device address
// is looked up once per device (with that device current) and cached.
// ---------------------------------------------------------------------------
static __device__ int g_dev_err;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
int *g_err_addr[kMaxDevices] = {};

int device_error_ptr(int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GDN_EUNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dev_err);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        g_err_addr[dev] = static_cast<int *>(p);
    }
    *out = g_err_addr[dev];
    return GDN_OK;
}

} // namespace

// ---------------------------------------------------------------------------
// Work counters of the state kernels.  Each state pool handle holds one pair
// (the next unit to claim, producers done) in this table, handed out on the
// host when the handle is made, so no call allocates device memory for it.
// The kernels leave a pair at zero when their launch ends; the table starts
// at zero when the module loads.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned int g_work[GDN_MAX_POOLS][2];

namespace {

std::mutex g_work_mu;
std::vector<int> g_work_free;
int g_work_next = 0;
unsigned int *g_work_addr[kMaxDevices] = {};

int work_index_take(int *index)
{
    std::lock_guard<std::mutex> lk(g_work_mu);
    if (!g_work_free.empty()) {
        *index = g_work_free.back();
        g_work_free.pop_back();
        return GDN_OK;
    }
    if (g_work_next >= GDN_MAX_POOLS)
        return fail(GDN_ENOMEM, "more than %d state pools alive at once", GDN_MAX_POOLS);
    *index = g_work_next++;
    return GDN_OK;
}

void work_index_give(int index)
{
    std::lock_guard<std::mutex> lk(g_work_mu);
    g_work_free.push_back(index);
}

// Device address of the pool's counter pair on the current device.
int work_ptr(const gdn_pool *pool, unsigned int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GDN_EUNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_work_mu);
    if (!g_work_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_work);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(work counters)");
        g_work_addr[dev] = static_cast<unsigned int *>(p);
    }
    *out = g_work_addr[dev] + 2 * (size_t)pool->work_index;
    return GDN_OK;
}

} // namespace

// ---------------------------------------------------------------------------
// small kernels
// ---------------------------------------------------------------------------
namespace {

__global__ void commit_kernel(int32_t *rs, int32_t *ws, int rows)
{
    gdn::wait_prior_grid();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < rows) {
        const int32_t t = rs[r];
        rs[r] = ws[r];
        ws[r] = t;
    }
}

// Zero whole slots of a pool whose slot is `slot_bytes` bytes (a multiple of 16).
__global__ void zero_slots_kernel(char *base, size_t slot_bytes, int num_slots, const int32_t *slots,
                                  int n, int *err)
{
    const size_t vec_per_slot = slot_bytes / 16;
    const size_t total = vec_per_slot * (size_t)n;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int k = (int)(i / vec_per_slot);
        const int s = slots[k];
        if (s < 0 || s >= num_slots) {
            if (i % vec_per_slot == 0)
                gdn::report(err, GDN_DEVERR_BAD_SLOT);
            continue;
        }
        reinterpret_cast<uint4 *>(base + (size_t)s * slot_bytes)[i % vec_per_slot] = make_uint4(0, 0, 0, 0);
    }
}

// Snapshots and forks: slot dst[k] receives slot src[k] of a pool whose slot
// is `slot_bytes` bytes (a multiple of 16).  A source outside the pool or a
// destination outside [1, num_slots) skips the pair and reports it.
__global__ void copy_slots_kernel(char *base, size_t slot_bytes, int num_slots, const int32_t *src,
                                  const int32_t *dst, int n, int *err)
{
    const size_t vec_per_slot = slot_bytes / 16;
    const size_t total = vec_per_slot * (size_t)n;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int k = (int)(i / vec_per_slot);
        const int s = src[k], d = dst[k];
        if (s < 0 || s >= num_slots || d <= 0 || d >= num_slots) {
            if (i % vec_per_slot == 0)
                gdn::report(err, GDN_DEVERR_BAD_SLOT);
            continue;
        }
        const uint4 v = reinterpret_cast<const uint4 *>(base + (size_t)s * slot_bytes)[i % vec_per_slot];
        reinterpret_cast<uint4 *>(base + (size_t)d * slot_bytes)[i % vec_per_slot] = v;
    }
}

// Traffic probes: the state bytes of a step, no arithmetic.  A block moves
// 16 KiB (4 vectors a thread), the size of one block of the state kernel at
// one pass with dk = 128.
constexpr int kProbeThreads = 256;
constexpr int kProbeFloats = kProbeThreads * 16;

__global__ void __launch_bounds__(kProbeThreads)
probe_kernel(float *pool, int num_slots, int hv, size_t head_floats, int chunks, const int32_t *rs_tab,
             const int32_t *ws_tab, int mode, float *sink, int *err)
{
    const int chunk = blockIdx.x % chunks;
    const int rh = blockIdx.x / chunks;
    const int h = rh % hv, r = rh / hv;
    const int rs = rs_tab[r];
    const bool in_place = mode == GDN_PROBE_INPLACE || mode == GDN_PROBE_READ;
    const int ws = in_place ? rs : ws_tab[r];
    const int cls = gdn::classify_row(rs, ws, num_slots, in_place);
    if (cls != 1) {
        if (cls < 0 && threadIdx.x == 0)
            gdn::report(err, GDN_DEVERR_BAD_SLOT);
        return;
    }
    const size_t off = (size_t)chunk * kProbeFloats;
    const float *src = pool + ((size_t)rs * hv + h) * head_floats + off;
    float *dst = pool + ((size_t)ws * hv + h) * head_floats + off;
    const size_t lim = head_floats - off < (size_t)kProbeFloats ? head_floats - off : kProbeFloats;
    float4 v[4];
    if (mode != GDN_PROBE_WRITE) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const size_t e = (size_t)(threadIdx.x + kProbeThreads * m) * 4;
            v[m] = e < lim ? gdn::ld_state(src + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    } else {
#pragma unroll
        for (int m = 0; m < 4; ++m)
            v[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (mode == GDN_PROBE_READ) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            acc += v[m].x + v[m].y + v[m].z + v[m].w;
        // the comparison keeps the loads alive; sink is practically never written
        if (acc == 123456.789f && sink)
            sink[(size_t)r * hv + h] = acc;
        return;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const size_t e = (size_t)(threadIdx.x + kProbeThreads * m) * 4;
        if (e < lim)
            gdn::st_state(dst + e, v[m]);
    }
}

} // namespace

// ---------------------------------------------------------------------------
// public API
// ---------------------------------------------------------------------------
extern "C" {

const char *gdn_last_error(void) { return t_msg; }

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

// ---- state pool -----------------------------------------------------------

static int check_dims(gdn_dims d)
{
    if (d.hk <= 0 || d.hv <= 0 || d.hv % d.hk != 0)
        return fail(GDN_EINVAL, "bad heads hk=%d hv=%d (need hv %% hk == 0)", d.hk, d.hv);
    if (!gdn::step_shape_supported(d.dk, d.dv))
        return fail(GDN_EUNSUPPORTED, "unsupported head dims dk=%d dv=%d", d.dk, d.dv);
    return GDN_OK;
}

static size_t state_slot_floats(gdn_dims d) { return (size_t)d.hv * d.dv * d.dk; }

// in-place counters: one 32-bit counter per (slot, qk head), a slot's row
// padded to 16 bytes so that zero_slots can clear it
static int qk_stride_of(gdn_dims d) { return (d.hk + 3) & ~3; }
static size_t qk_count_bytes(int num_slots, gdn_dims d)
{
    return (size_t)num_slots * (size_t)qk_stride_of(d) * sizeof(unsigned int);
}

int gdn_state_pool_create(int num_slots, gdn_dims dims, void *stream, gdn_pool **out)
{
    if (!out)
        return fail(GDN_EINVAL, "out is NULL");
    *out = nullptr;
    if (num_slots < 1)
        return fail(GDN_EINVAL, "num_slots=%d < 1", num_slots);
    int rc = check_dims(dims);
    if (rc)
        return rc;
    const size_t bytes = state_slot_floats(dims) * sizeof(float) * (size_t)num_slots;
    void *p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e == cudaErrorMemoryAllocation) {
        cudaGetLastError();
        return fail(GDN_ENOMEM, "cudaMalloc(%zu bytes) for the state pool failed", bytes);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(state pool)");
    const size_t cbytes = qk_count_bytes(num_slots, dims);
    void *cnt = nullptr;
    e = cudaMalloc(&cnt, cbytes);
    if (e != cudaSuccess) {
        cudaFree(p);
        if (e == cudaErrorMemoryAllocation) {
            cudaGetLastError();
            return fail(GDN_ENOMEM, "cudaMalloc(%zu bytes) for the in-place counters failed", cbytes);
        }
        return cuda_fail(e, "cudaMalloc(in-place counters)");
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(p, 0, bytes, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(cnt, 0, cbytes, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaFree(p);
        cudaFree(cnt);
        return cuda_fail(e, "zero-filling the state pool");
    }
    int wi = 0;
    rc = work_index_take(&wi);
    if (rc) {
        cudaFree(p);
        cudaFree(cnt);
        return rc;
    }
    *out = new gdn_pool{static_cast<float *>(p), num_slots, dims, true, wi,
                        static_cast<unsigned int *>(cnt), qk_stride_of(dims), true};
    return ok();
}

int gdn_state_pool_wrap(void *dev_ptr, int num_slots, gdn_dims dims, gdn_pool **out)
{
    if (!out)
        return fail(GDN_EINVAL, "out is NULL");
    *out = nullptr;
    if (!dev_ptr)
        return fail(GDN_EINVAL, "dev_ptr is NULL");
    if (!aligned16(dev_ptr))
        return fail(GDN_EINVAL, "state pool memory must be 16-byte aligned");
    if (num_slots < 1)
        return fail(GDN_EINVAL, "num_slots=%d < 1", num_slots);
    int rc = check_dims(dims);
    if (rc)
        return rc;
    int wi = 0;
    rc = work_index_take(&wi);
    if (rc)
        return rc;
    *out = new gdn_pool{static_cast<float *>(dev_ptr), num_slots, dims, false, wi, nullptr, qk_stride_of(dims),
                        false};
    return ok();
}

size_t gdn_pool_inplace_counter_bytes(int num_slots, gdn_dims dims)
{
    if (num_slots < 1 || check_dims(dims) != GDN_OK)
        return 0;
    return qk_count_bytes(num_slots, dims);
}

int gdn_pool_attach_inplace_counters(gdn_pool *pool, void *dev_counters, size_t bytes)
{
    if (!pool)
        return fail(GDN_EINVAL, "pool is NULL");
    if (pool->owns_qk_count)
        return fail(GDN_EINVAL, "the pool was created with its own in-place counters");
    if (!dev_counters) {
        pool->qk_count = nullptr;
        return ok();
    }
    if (!aligned16(dev_counters))
        return fail(GDN_EINVAL, "in-place counters must be 16-byte aligned");
    const size_t need = qk_count_bytes(pool->num_slots, pool->dims);
    if (bytes < need)
        return fail(GDN_EINVAL, "in-place counters of %zu bytes: the pool needs %zu", bytes, need);
    pool->qk_count = static_cast<unsigned int *>(dev_counters);
    return ok();
}

int gdn_state_pool_destroy(gdn_pool *pool)
{
    if (!pool)
        return ok();
    cudaError_t e = cudaSuccess;
    if (pool->owned)
        e = cudaFree(pool->data);
    if (pool->owns_qk_count) {
        const cudaError_t e2 = cudaFree(pool->qk_count);
        if (e == cudaSuccess)
            e = e2;
    }
    work_index_give(pool->work_index);
    delete pool;
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFree(state pool)");
    return ok();
}

void *gdn_pool_data(const gdn_pool *pool) { return pool ? pool->data : nullptr; }
int gdn_pool_num_slots(const gdn_pool *pool) { return pool ? pool->num_slots : 0; }
gdn_dims gdn_pool_dims(const gdn_pool *pool)
{
    gdn_dims z = {0, 0, 0, 0};
    return pool ? pool->dims : z;
}

static int zero_slots(void *base, size_t slot_bytes, int num_slots, const int32_t *slots, int n,
                      void *stream)
{
    if (n < 0)
        return fail(GDN_EINVAL, "n=%d < 0", n);
    if (n == 0)
        return ok();
    if (!slots)
        return fail(GDN_EINVAL, "slots is NULL");
    int *err = nullptr;
    int rc = device_error_ptr(&err);
    if (rc)
        return rc;
    const size_t total = slot_bytes / 16 * (size_t)n;
    size_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16)
        blocks = 152 * 16;
    zero_slots_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<char *>(base), slot_bytes, num_slots, slots, n, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "zero_slots launch");
    return ok();
}

static int copy_slots(void *base, size_t slot_bytes, int num_slots, const int32_t *src, const int32_t *dst,
                      int n, void *stream)
{
    if (n < 0)
        return fail(GDN_EINVAL, "n=%d < 0", n);
    if (n == 0)
        return ok();
    if (!src || !dst)
        return fail(GDN_EINVAL, "src and dst must be non-NULL");
    int *err = nullptr;
    int rc = device_error_ptr(&err);
    if (rc)
        return rc;
    const size_t total = slot_bytes / 16 * (size_t)n;
    size_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16)
        blocks = 152 * 16;
    copy_slots_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<char *>(base), slot_bytes, num_slots, src, dst, n, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "copy_slots launch");
    return ok();
}

int gdn_pool_copy_slots(gdn_pool *pool, const int32_t *src, const int32_t *dst, int n, void *stream)
{
    if (!pool)
        return fail(GDN_EINVAL, "pool is NULL");
    return copy_slots(pool->data, state_slot_floats(pool->dims) * sizeof(float), pool->num_slots, src, dst, n,
                      stream);
}

int gdn_pool_zero_slots(gdn_pool *pool, const int32_t *slots, int n, void *stream)
{
    if (!pool)
        return fail(GDN_EINVAL, "pool is NULL");
    int rc = zero_slots(pool->data, state_slot_floats(pool->dims) * sizeof(float), pool->num_slots, slots, n,
                        stream);
    if (rc || !pool->qk_count)
        return rc;
    // the slots' in-place counters too (a launch that stopped early can leave them set)
    return zero_slots(pool->qk_count, (size_t)pool->qk_stride * sizeof(unsigned int), pool->num_slots, slots, n,
                      stream);
}

// ---- conv pool -------------------------------------------------------------

static int check_conv_geometry(int num_slots, int channels, int width, int dtype)
{
    if (num_slots < 1)
        return fail(GDN_EINVAL, "num_slots=%d < 1", num_slots);
    if (channels <= 0 || channels % 8 != 0)
        return fail(GDN_EINVAL, "channels=%d must be a positive multiple of 8", channels);
    if (width < 2 || width > 4)
        return fail(GDN_EUNSUPPORTED, "conv width %d not in 2..4", width);
    if (!dtype_ok(dtype))
        return fail(GDN_EINVAL, "bad dtype %d", dtype);
    return GDN_OK;
}

int conv_state_pool_create(int num_slots, int channels, int width, int dtype, void *stream,
                           conv_pool **out)
{
    if (!out)
        return fail(GDN_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = check_conv_geometry(num_slots, channels, width, dtype);
    if (rc)
        return rc;
    const size_t bytes = (size_t)num_slots * (width - 1) * channels * dtype_size(dtype);
    void *p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e == cudaErrorMemoryAllocation) {
        cudaGetLastError();
        return fail(GDN_ENOMEM, "cudaMalloc(%zu bytes) for the conv pool failed", bytes);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(conv pool)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(p, 0, bytes, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_fail(e, "zero-filling the conv pool");
    }
    *out = new conv_pool{p, num_slots, channels, width, dtype, true};
    return ok();
}

int conv_state_pool_wrap(void *dev_ptr, int num_slots, int channels, int width, int dtype,
                         conv_pool **out)
{
    if (!out)
        return fail(GDN_EINVAL, "out is NULL");
    *out = nullptr;
    if (!dev_ptr)
        return fail(GDN_EINVAL, "dev_ptr is NULL");
    if (!aligned16(dev_ptr))
        return fail(GDN_EINVAL, "conv pool memory must be 16-byte aligned");
    int rc = check_conv_geometry(num_slots, channels, width, dtype);
    if (rc)
        return rc;
    *out = new conv_pool{dev_ptr, num_slots, channels, width, dtype, false};
    return ok();
}

int conv_state_pool_destroy(conv_pool *pool)
{
    if (!pool)
        return ok();
    cudaError_t e = cudaSuccess;
    if (pool->owned)
        e = cudaFree(pool->data);
    delete pool;
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFree(conv pool)");
    return ok();
}

void *conv_pool_data(const conv_pool *pool) { return pool ? pool->data : nullptr; }
int conv_pool_num_slots(const conv_pool *pool) { return pool ? pool->num_slots : 0; }

int conv_pool_copy_slots(conv_pool *pool, const int32_t *src, const int32_t *dst, int n, void *stream)
{
    if (!pool)
        return fail(GDN_EINVAL, "pool is NULL");
    return copy_slots(pool->data, (size_t)(pool->width - 1) * pool->channels * dtype_size(pool->dtype),
                      pool->num_slots, src, dst, n, stream);
}

int conv_pool_zero_slots(conv_pool *pool, const int32_t *slots, int n, void *stream)
{
    if (!pool)
        return fail(GDN_EINVAL, "pool is NULL");
    const size_t slot_bytes = (size_t)(pool->width - 1) * pool->channels * dtype_size(pool->dtype);
    return zero_slots(pool->data, slot_bytes, pool->num_slots, slots, n, stream);
}

// ---- causal_conv1d_decode ---------------------------------------------------

int causal_conv1d_decode(const void *x, int x_row_stride, conv_pool *cp, const int32_t *slot_idx,
                         const int32_t *write_slot, const void *w, const void *bias, int silu,
                         void *out, int rows, int dtype, void *stream)
{
    if (!cp)
        return fail(GDN_EINVAL, "conv pool is NULL");
    if (rows < 0)
        return fail(GDN_EINVAL, "rows=%d < 0", rows);
    if (!dtype_ok(dtype) || dtype != cp->dtype)
        return fail(GDN_EINVAL, "dtype %d does not match the conv pool's %d", dtype, cp->dtype);
    if (rows == 0)
        return ok();
    if (!x || !slot_idx || !w || !out)
        return fail(GDN_EINVAL, "x, slot_idx, w and out must be non-NULL");
    if (x_row_stride < cp->channels || x_row_stride % 8 != 0)
        return fail(GDN_EINVAL, "x_row_stride=%d must be >= channels (%d) and a multiple of 8",
                    x_row_stride, cp->channels);
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || (bias && !aligned16(bias)))
        return fail(GDN_EINVAL, "x, w, bias and out must be 16-byte aligned");
    int *err = nullptr;
    int rc = device_error_ptr(&err);
    if (rc)
        return rc;
    gdn::ConvArgs a;
    a.x = x;
    a.x_stride = x_row_stride;
    a.conv = cp->data;
    a.num_slots = cp->num_slots;
    a.read_slot = slot_idx;
    a.write_slot = write_slot;
    a.w = w;
    a.bias = bias;
    a.silu = silu ? 1 : 0;
    a.out = out;
    a.rows = rows;
    a.channels = cp->channels;
    a.width = cp->width;
    a.err = err;
    cudaError_t e = gdn::launch_conv(a, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "causal_conv1d_decode launch");
    return ok();
}

// ---- gdn_decode_step / gdn_layer_decode --------------------------------------

static int check_state_common(gdn_pool *pool, const void *a, const void *b, const float *A_log,
                              const float *dt_bias, const int32_t *read_slot, const int32_t *write_slot,
                              const void *out, int rows, int keep_in_place, int dtype)
{
    if (!pool)
        return fail(GDN_EINVAL, "state pool is NULL");
    if (rows < 0)
        return fail(GDN_EINVAL, "rows=%d < 0", rows);
    if (!dtype_ok(dtype))
        return fail(GDN_EINVAL, "bad dtype %d", dtype);
    if (rows == 0)
        return GDN_OK;
    if (!a || !b || !A_log || !dt_bias || !read_slot || !out)
        return fail(GDN_EINVAL, "a, b, A_log, dt_bias, read_slot and out must be non-NULL");
    if (!keep_in_place && !write_slot)
        return fail(GDN_EINVAL, "write_slot is NULL in twin mode");
    return GDN_OK;
}

int gdn_decode_step(const void *q, const void *k, const void *v, const void *a, const void *b,
                    const float *A_log, const float *dt_bias, gdn_pool *pool,
                    const int32_t *read_slot, const int32_t *write_slot, void *out, int rows,
                    int heads, int keep_in_place, int dtype, void *stream)
{
    int rc = check_state_common(pool, a, b, A_log, dt_bias, read_slot, write_slot, out, rows,
                                keep_in_place, dtype);
    if (rc)
        return rc;
    if (heads != pool->dims.hv)
        return fail(GDN_EINVAL, "heads=%d differs from the pool's hv=%d", heads, pool->dims.hv);
    if (rows == 0)
        return ok();
    if (!q || !k || !v)
        return fail(GDN_EINVAL, "q, k and v must be non-NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v))
        return fail(GDN_EINVAL, "q, k and v must be 16-byte aligned");
    int *err = nullptr;
    rc = device_error_ptr(&err);
    if (rc)
        return rc;
    gdn::StepArgs s = {};
    s.q = q;
    s.k = k;
    s.v = v;
    s.a = a;
    s.b = b;
    s.A_log = A_log;
    s.dt_bias = dt_bias;
    s.pool = pool->data;
    s.num_slots = pool->num_slots;
    s.read_slot = read_slot;
    s.write_slot = write_slot;
    s.in_place = keep_in_place ? 1 : 0;
    s.out = out;
    s.rows = rows;
    s.hk = pool->dims.hk;
    s.hv = pool->dims.hv;
    s.dk = pool->dims.dk;
    s.dv = pool->dims.dv;
    s.err = err;
    rc = work_ptr(pool, &s.work);
    if (rc)
        return rc;
    cudaError_t e = gdn::launch_gdn_step(s, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_decode_step launch");
    return ok();
}

// Checks a fused layer call and fills its launch arguments, all but the work
// counters.  *none is set when there is nothing to launch (rows == 0).
static int layer_args(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                      const float *A_log, const float *dt_bias, const void *a, const void *b,
                      gdn_pool *pool, const int32_t *read_slot, const int32_t *write_slot, void *out,
                      int rows, int keep_in_place, int dtype, gdn::StepArgs *s, bool *none)
{
    *none = true;
    int rc = check_state_common(pool, a, b, A_log, dt_bias, read_slot, write_slot, out, rows,
                                keep_in_place, dtype);
    if (rc)
        return rc;
    if (!cp)
        return fail(GDN_EINVAL, "conv pool is NULL");
    const gdn_dims d = pool->dims;
    const int C = 2 * d.hk * d.dk + d.hv * d.dv;
    if (cp->channels != C)
        return fail(GDN_EINVAL, "conv pool has %d channels, the layer needs 2*hk*dk + hv*dv = %d",
                    cp->channels, C);
    if (cp->dtype != dtype)
        return fail(GDN_EINVAL, "dtype %d does not match the conv pool's %d", dtype, cp->dtype);
    if (!gdn::layer_shape_supported(d.dk, d.dv, d.hv / d.hk, keep_in_place != 0))
        return fail(GDN_EUNSUPPORTED, "unsupported layer shape (hv/hk=%d, dk=%d, dv=%d)", d.hv / d.hk,
                    d.dk, d.dv);
    if (rows == 0)
        return ok();
    if (!x || !w)
        return fail(GDN_EINVAL, "x and w must be non-NULL");
    if (!aligned16(x) || !aligned16(w) || (bias && !aligned16(bias)))
        return fail(GDN_EINVAL, "x, w and bias must be 16-byte aligned");
    int *err = nullptr;
    rc = device_error_ptr(&err);
    if (rc)
        return rc;
    *s = gdn::StepArgs{};
    s->a = a;
    s->b = b;
    s->A_log = A_log;
    s->dt_bias = dt_bias;
    s->pool = pool->data;
    s->num_slots = pool->num_slots < cp->num_slots ? pool->num_slots : cp->num_slots;
    s->read_slot = read_slot;
    s->write_slot = write_slot;
    s->in_place = keep_in_place ? 1 : 0;
    s->qk_count = keep_in_place ? pool->qk_count : nullptr;
    s->qk_stride = pool->qk_stride;
    s->out = out;
    s->rows = rows;
    s->hk = d.hk;
    s->hv = d.hv;
    s->dk = d.dk;
    s->dv = d.dv;
    s->err = err;
    s->x = x;
    s->conv = cp->data;
    s->w = w;
    s->bias = bias;
    s->silu = silu ? 1 : 0;
    s->width = cp->width;
    s->channels = C;
    *none = false;
    return GDN_OK;
}

int gdn_layer_decode(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                     const float *A_log, const float *dt_bias, const void *a, const void *b,
                     gdn_pool *pool, const int32_t *read_slot, const int32_t *write_slot,
                     void *out, int rows, int keep_in_place, int dtype, void *stream)
{
    gdn::StepArgs s;
    bool none = true;
    int rc = layer_args(x, cp, w, bias, silu, A_log, dt_bias, a, b, pool, read_slot, write_slot, out,
                        rows, keep_in_place, dtype, &s, &none);
    if (rc || none)
        return rc;
    rc = work_ptr(pool, &s.work);
    if (rc)
        return rc;
    cudaError_t e = gdn::launch_gdn_layer(s, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_layer_decode launch");
    return ok();
}

int gdn_layer_decode_commit(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                            const float *A_log, const float *dt_bias, const void *a, const void *b,
                            gdn_pool *pool, int32_t *read_slot, int32_t *write_slot, void *out,
                            int rows, int dtype, void *stream)
{
    gdn::StepArgs s;
    bool none = true;
    int rc = layer_args(x, cp, w, bias, silu, A_log, dt_bias, a, b, pool, read_slot, write_slot, out,
                        rows, 0, dtype, &s, &none);
    if (rc || none)
        return rc;
    rc = work_ptr(pool, &s.work);
    if (rc)
        return rc;
    s.commit = 1;
    cudaError_t e = gdn::launch_gdn_layer(s, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_layer_decode_commit launch");
    return ok();
}

// ---- many tokens a sequence: gdn_prefill, gdn_verify, causal_conv1d_prefill ------

static int check_tokens(int nseq, int total_tokens, const int32_t *cu_seqlens, const int32_t *read_slot,
                        int dtype)
{
    if (nseq < 0 || total_tokens < 0)
        return fail(GDN_EINVAL, "nseq=%d and total_tokens=%d must be >= 0", nseq, total_tokens);
    if (!dtype_ok(dtype))
        return fail(GDN_EINVAL, "bad dtype %d", dtype);
    if (nseq > 0 && (!cu_seqlens || !read_slot))
        return fail(GDN_EINVAL, "cu_seqlens and read_slot must be non-NULL");
    return GDN_OK;
}

static int prefill_launch(const void *q, const void *k, const void *v, const void *a, const void *b,
                          const float *A_log, const float *dt_bias, gdn_pool *pool, const int32_t *cu_seqlens,
                          const int32_t *read_slot, const int32_t *write_slot, const int32_t *token_slot,
                          void *out, int nseq, int total_tokens, int dtype, void *stream, const char *what,
                          bool chunked = false, void *work = nullptr)
{
    if (!pool)
        return fail(GDN_EINVAL, "state pool is NULL");
    int rc = check_tokens(nseq, total_tokens, cu_seqlens, read_slot, dtype);
    if (rc)
        return rc;
    if (nseq == 0)
        return ok();
    if (total_tokens > 0) {
        if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !out)
            return fail(GDN_EINVAL, "q, k, v, a, b, A_log, dt_bias and out must be non-NULL");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v))
            return fail(GDN_EINVAL, "q, k and v must be 16-byte aligned");
    }
    int *err = nullptr;
    rc = device_error_ptr(&err);
    if (rc)
        return rc;
    gdn::PrefillArgs s = {};
    s.q = q;
    s.k = k;
    s.v = v;
    s.a = a;
    s.b = b;
    s.A_log = A_log;
    s.dt_bias = dt_bias;
    s.pool = pool->data;
    s.num_slots = pool->num_slots;
    s.cu_seqlens = cu_seqlens;
    s.read_slot = read_slot;
    s.write_slot = write_slot;
    s.token_slot = token_slot;
    s.out = out;
    s.nseq = nseq;
    s.total_tokens = total_tokens;
    s.hk = pool->dims.hk;
    s.hv = pool->dims.hv;
    s.dk = pool->dims.dk;
    s.dv = pool->dims.dv;
    s.err = err;
    s.work = work;
    cudaError_t e = chunked ? gdn::launch_gdn_prefill_chunked(s, dtype, static_cast<cudaStream_t>(stream))
                            : gdn::launch_gdn_prefill(s, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, what);
    return ok();
}

int gdn_prefill(const void *q, const void *k, const void *v, const void *a, const void *b,
                const float *A_log, const float *dt_bias, gdn_pool *pool, const int32_t *cu_seqlens,
                const int32_t *read_slot, const int32_t *write_slot, void *out, int nseq, int total_tokens,
                int keep_in_place, int dtype, void *stream)
{
    if (!keep_in_place && nseq > 0 && !write_slot)
        return fail(GDN_EINVAL, "write_slot is NULL in twin mode");
    return prefill_launch(q, k, v, a, b, A_log, dt_bias, pool, cu_seqlens, read_slot,
                          keep_in_place ? nullptr : write_slot, nullptr, out, nseq, total_tokens, dtype,
                          stream, "gdn_prefill launch");
}

size_t gdn_prefill_chunked_workspace_bytes(int nseq, int total_tokens, int hv)
{
    return gdn::prefill_chunked_workspace_bytes(nseq, total_tokens, hv);
}

int gdn_prefill_chunked(const void *q, const void *k, const void *v, const void *a, const void *b,
                        const float *A_log, const float *dt_bias, gdn_pool *pool, const int32_t *cu_seqlens,
                        const int32_t *read_slot, const int32_t *write_slot, void *out, int nseq,
                        int total_tokens, int keep_in_place, void *workspace, size_t workspace_bytes, int dtype,
                        void *stream)
{
    if (pool && !gdn::chunked_shape_supported(pool->dims.dk, pool->dims.dv))
        return fail(GDN_EUNSUPPORTED, "gdn_prefill_chunked is built for dk = dv = 128 (pool has %d, %d)",
                    pool->dims.dk, pool->dims.dv);
    if (!keep_in_place && nseq > 0 && !write_slot)
        return fail(GDN_EINVAL, "write_slot is NULL in twin mode");
    if (pool && dtype == GDN_BF16 && nseq > 0) {
        const size_t need = gdn::prefill_chunked_workspace_bytes(nseq, total_tokens, pool->dims.hv);
        if (!workspace || workspace_bytes < need)
            return fail(GDN_EINVAL, "workspace of %zu bytes at %p: bf16 activations need %zu bytes", workspace_bytes,
                        workspace, need);
        if ((reinterpret_cast<uintptr_t>(workspace) & 127u) != 0)
            return fail(GDN_EINVAL, "workspace must be 128-byte aligned");
    }
    return prefill_launch(q, k, v, a, b, A_log, dt_bias, pool, cu_seqlens, read_slot,
                          keep_in_place ? nullptr : write_slot, nullptr, out, nseq, total_tokens, dtype,
                          stream, "gdn_prefill_chunked launch", true, workspace);
}

int gdn_verify(const void *q, const void *k, const void *v, const void *a, const void *b,
               const float *A_log, const float *dt_bias, gdn_pool *pool, const int32_t *cu_seqlens,
               const int32_t *read_slot, const int32_t *token_slot, void *out, int nseq, int total_tokens,
               int dtype, void *stream)
{
    if (!pool)
        return fail(GDN_EINVAL, "state pool is NULL");
    int rc = check_tokens(nseq, total_tokens, cu_seqlens, read_slot, dtype);
    if (rc)
        return rc;
    if (nseq == 0 || total_tokens == 0)
        return ok(); // no token, no state to keep
    if (!token_slot)
        return fail(GDN_EINVAL, "token_slot must be non-NULL");
    return prefill_launch(q, k, v, a, b, A_log, dt_bias, pool, cu_seqlens, read_slot, nullptr, token_slot,
                          out, nseq, total_tokens, dtype, stream, "gdn_verify launch");
}

int causal_conv1d_prefill(const void *x, conv_pool *cp, const int32_t *cu_seqlens, const int32_t *read_slot,
                          const int32_t *write_slot, const int32_t *token_slot, const void *w,
                          const void *bias, int silu, void *out, int nseq, int total_tokens, int dtype,
                          void *stream)
{
    if (!cp)
        return fail(GDN_EINVAL, "conv pool is NULL");
    int rc = check_tokens(nseq, total_tokens, cu_seqlens, read_slot, dtype);
    if (rc)
        return rc;
    if (dtype != cp->dtype)
        return fail(GDN_EINVAL, "dtype %d does not match the conv pool's %d", dtype, cp->dtype);
    if (nseq == 0)
        return ok();
    if (!w || (total_tokens > 0 && (!x || !out)))
        return fail(GDN_EINVAL, "x, w and out must be non-NULL");
    if ((x && !aligned16(x)) || !aligned16(w) || (out && !aligned16(out)) || (bias && !aligned16(bias)))
        return fail(GDN_EINVAL, "x, w, bias and out must be 16-byte aligned");
    int *err = nullptr;
    rc = device_error_ptr(&err);
    if (rc)
        return rc;
    gdn::ConvPrefillArgs s = {};
    s.x = x;
    s.conv = cp->data;
    s.num_slots = cp->num_slots;
    s.cu_seqlens = cu_seqlens;
    s.read_slot = read_slot;
    s.write_slot = write_slot;
    s.token_slot = token_slot;
    s.w = w;
    s.bias = bias;
    s.silu = silu ? 1 : 0;
    s.out = out;
    s.nseq = nseq;
    s.total_tokens = total_tokens;
    s.channels = cp->channels;
    s.width = cp->width;
    s.err = err;
    cudaError_t e = gdn::launch_conv_prefill(s, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "causal_conv1d_prefill launch");
    return ok();
}

int gdn_layer_decode_bucket(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                            const float *A_log, const float *dt_bias, const void *a, const void *b,
                            gdn_pool *pool, int32_t *read_slot, int32_t *write_slot, void *out, int rows,
                            const int32_t *n_decode, int keep_in_place, int commit, int dtype, void *stream)
{
    if (commit && keep_in_place)
        return fail(GDN_EINVAL, "commit swaps twin slots; it does not apply in place");
    if (rows > 0 && !n_decode)
        return fail(GDN_EINVAL, "n_decode is NULL");
    gdn::StepArgs s;
    bool none = true;
    int rc = layer_args(x, cp, w, bias, silu, A_log, dt_bias, a, b, pool, read_slot, write_slot, out, rows,
                        keep_in_place, dtype, &s, &none);
    if (rc || none)
        return rc;
    rc = work_ptr(pool, &s.work);
    if (rc)
        return rc;
    s.n_live = n_decode;
    s.commit = commit ? 1 : 0;
    cudaError_t e = gdn::launch_gdn_layer(s, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_layer_decode_bucket launch");
    return ok();
}

// ---- gdn_layer_decode_noalloc ------------------------------------------------
// gdn_layer_decode for callers that cannot allocate device memory: the work
// counters of the launch come from a fixed array of this file, looked up once
// per device, instead of the state pool's pair.

static __device__ __align__(256) unsigned int g_noalloc_scratch[GDN_NOALLOC_SCRATCH_SLOTS][2];

namespace {

std::mutex g_noalloc_mu;
unsigned int *g_noalloc_addr[kMaxDevices] = {};

int noalloc_scratch_ptr(unsigned int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GDN_EUNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        unsigned int *p = nullptr;
        e = cudaGetSymbolAddress((void **)&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return GDN_OK;
}

} // namespace

int gdn_layer_decode_noalloc(const void *x, conv_pool *cp, const void *w, const void *bias, int silu,
                             const float *A_log, const float *dt_bias, const void *a, const void *b,
                             gdn_pool *pool, const int32_t *read_slot, const int32_t *write_slot,
                             void *out, int rows, int keep_in_place, int scratch_slot, int dtype,
                             void *stream)
{
    if (scratch_slot < 0 || scratch_slot >= GDN_NOALLOC_SCRATCH_SLOTS)
        return fail(GDN_EINVAL,
                    "scratch_slot=%d: the no-allocation scratch holds %d slots of %d bytes (%d bytes)",
                    scratch_slot, GDN_NOALLOC_SCRATCH_SLOTS, (int)(2 * sizeof(unsigned int)),
                    (int)sizeof(g_noalloc_scratch));
    gdn::StepArgs s;
    bool none = true;
    int rc = layer_args(x, cp, w, bias, silu, A_log, dt_bias, a, b, pool, read_slot, write_slot, out,
                        rows, keep_in_place, dtype, &s, &none);
    if (rc || none)
        return rc;
    unsigned int *scratch = nullptr;
    rc = noalloc_scratch_ptr(&scratch);
    if (rc)
        return rc;
    s.work = scratch + 2 * (size_t)scratch_slot;
    cudaError_t e = gdn::launch_gdn_layer(s, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_layer_decode_noalloc launch");
    return ok();
}

// ---- commit, validation, device errors ---------------------------------------

int gdn_commit(int32_t *read_slot, int32_t *write_slot, int rows, void *stream)
{
    if (rows < 0)
        return fail(GDN_EINVAL, "rows=%d < 0", rows);
    if (rows == 0)
        return ok();
    if (!read_slot || !write_slot)
        return fail(GDN_EINVAL, "slot tables must be non-NULL");
    cudaError_t e = gdn::launch_pdl(commit_kernel, dim3((rows + 255) / 256), dim3(256), 0,
                                    static_cast<cudaStream_t>(stream), read_slot, write_slot, rows);
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_commit launch");
    return ok();
}

int gdn_validate_slots(const int32_t *read_slot, const int32_t *write_slot, int rows, int num_slots,
                       int keep_in_place, void *stream)
{
    if (rows < 0 || num_slots < 1)
        return fail(GDN_EINVAL, "rows=%d num_slots=%d", rows, num_slots);
    if (rows == 0)
        return ok();
    if (!read_slot || (!keep_in_place && !write_slot))
        return fail(GDN_EINVAL, "slot tables must be non-NULL");
    std::vector<int32_t> rs(rows), ws(rows);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(rs.data(), read_slot, sizeof(int32_t) * rows, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && !keep_in_place)
        e = cudaMemcpyAsync(ws.data(), write_slot, sizeof(int32_t) * rows, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "copying slot tables");
    if (keep_in_place)
        ws = rs;
    std::vector<int> writer(num_slots, -1), reader(num_slots, -1);
    for (int r = 0; r < rows; ++r) {
        const int a = rs[r], b = ws[r];
        if (a < 0 || a >= num_slots)
            return fail(GDN_ESLOTS, "row %d: read slot %d outside [0, %d)", r, a, num_slots);
        if (a == 0)
            continue; // padding row
        if (b <= 0 || b >= num_slots)
            return fail(GDN_ESLOTS, "row %d: write slot %d outside [1, %d)", r, b, num_slots);
        if (!keep_in_place && a == b)
            return fail(GDN_ESLOTS, "row %d: twin write slot equals its read slot %d", r, a);
        if (reader[a] >= 0)
            return fail(GDN_ESLOTS, "rows %d and %d read slot %d", reader[a], r, a);
        reader[a] = r;
        if (writer[b] >= 0)
            return fail(GDN_ESLOTS, "rows %d and %d write slot %d", writer[b], r, b);
        writer[b] = r;
    }
    for (int s2 = 1; s2 < num_slots; ++s2)
        if (writer[s2] >= 0 && reader[s2] >= 0 && writer[s2] != reader[s2])
            return fail(GDN_ESLOTS, "row %d writes slot %d that row %d reads", writer[s2], s2, reader[s2]);
    return ok();
}

int gdn_get_device_error(int *code, void *stream)
{
    if (!code)
        return fail(GDN_EINVAL, "code is NULL");
    int *err = nullptr;
    int rc = device_error_ptr(&err);
    if (rc)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, err, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(err, 0, sizeof(int), s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the device error word");
    *code = h;
    return ok();
}

// ---- probes ----------------------------------------------------------------------

int gdn_probe_traffic(gdn_pool *pool, const int32_t *read_slot, const int32_t *write_slot, int rows,
                      int mode, float *sink, void *stream)
{
    if (!pool)
        return fail(GDN_EINVAL, "pool is NULL");
    if (mode < GDN_PROBE_TWIN || mode > GDN_PROBE_WRITE)
        return fail(GDN_EINVAL, "bad probe mode %d", mode);
    if (rows < 0)
        return fail(GDN_EINVAL, "rows=%d < 0", rows);
    if (rows == 0)
        return ok();
    const bool needs_ws = mode == GDN_PROBE_TWIN || mode == GDN_PROBE_WRITE;
    if (!read_slot || (needs_ws && !write_slot))
        return fail(GDN_EINVAL, "slot tables must be non-NULL");
    int *err = nullptr;
    int rc = device_error_ptr(&err);
    if (rc)
        return rc;
    const gdn_dims d = pool->dims;
    const size_t head_floats = (size_t)d.dv * d.dk;
    const int chunks = (int)((head_floats + kProbeFloats - 1) / kProbeFloats);
    const long long blocks = (long long)rows * d.hv * chunks;
    probe_kernel<<<(unsigned)blocks, kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        pool->data, pool->num_slots, d.hv, head_floats, chunks, read_slot, write_slot, mode, sink, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_probe_traffic launch");
    return ok();
}

} // extern "C"

namespace {

// A wait that nothing ends: one thread waits for the first phase of an
// mbarrier no thread arrives at, through the bounded wait every kernel uses
// (here with the caller's time limit), and reports the timeout in the device
// error word.  The failure path runs without anything faulting or hanging:
// no copy is in flight and the thread leaves normally.
__global__ void wait_selftest_kernel(int *err, unsigned long long limit_ns)
{
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = gdn::sm_addr(&bar);
    gdn::mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!gdn::mbar_wait(b, 0, limit_ns))
        gdn::report(err, GDN_DEVERR_TIMEOUT);
}

} // namespace

extern "C" {

int gdn_selftest_wait_timeout(int limit_us, void *stream)
{
    if (limit_us < 1 || (unsigned long long)limit_us * 1000ull > gdn::kWaitNs)
        return fail(GDN_EINVAL, "limit_us=%d outside [1, %llu]", limit_us, gdn::kWaitNs / 1000ull);
    int *err = nullptr;
    int rc = device_error_ptr(&err);
    if (rc)
        return rc;
    wait_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err, (unsigned long long)limit_us * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "gdn_selftest_wait_timeout launch");
    return ok();
}

} // extern "C"
