// api.cu - the C ABI of libtfk (include/tfk.h): host-side argument
// validation, status reporting and kernel launch.  Nothing here allocates,
// frees or synchronises.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/tfk.h"
#include "device_scope.h"
#include "kernels.h"
#include "status.h"

namespace tfk {

// ---- device attribute and occupancy caches ----------------------------------

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
std::atomic<bool> g_have[kMaxDevices];

struct OccEntry {
    int dev;
    const void* func;
    int threads;
    size_t smem;
    int blocks;
};
constexpr int kOccEntries = 128;
OccEntry g_occ[kOccEntries];
int g_occ_n = 0;
}  // namespace

cudaError_t device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_have[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_have[dev].load(std::memory_order_relaxed)) {
            DeviceInfo d{};
            if ((err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return err;
            if ((err = cudaDeviceGetAttribute(&d.max_smem_per_block_optin,
                                              cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
                return err;
            if ((err = cudaDeviceGetAttribute(&d.max_smem_per_sm,
                                              cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
                return err;
            g_info[dev] = d;
            g_have[dev].store(true, std::memory_order_release);
        }
    }
    *out = g_info[dev];
    return cudaSuccess;
}

int blocks_per_sm(const void* func, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_occ_n; ++i) {
        const OccEntry& e = g_occ[i];
        if (e.dev == dev && e.func == func && e.threads == threads && e.smem == smem) return e.blocks;
    }
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, func) != cudaSuccess) {
        cudaGetLastError();  // leave no stale error for the next launch check
        return 0;
    }
    if (smem + fa.sharedSizeBytes > 48 * 1024) {  // beyond the default limit, static shared memory included
        // always the device maximum, so that launches of other sizes never lower it
        DeviceInfo di;
        if (g_have[dev].load(std::memory_order_acquire)) {
            di = g_info[dev];
        } else {
            int optin = 0;
            if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
            di.max_smem_per_block_optin = optin;
        }
        const int64_t dyn_max = (int64_t)di.max_smem_per_block_optin - (int64_t)fa.sharedSizeBytes;
        if ((int64_t)smem > dyn_max) return 0;
        if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_max) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
    }
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, func, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (g_occ_n < kOccEntries) g_occ[g_occ_n++] = OccEntry{dev, func, threads, smem, blocks};
    return blocks;
}

int pick_stages(int ctas_per_sm, int stage_bytes, int extra_bytes, int inflight_per_sm) {
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess || stage_bytes <= 0) return 2;
    if (ctas_per_sm < 1) ctas_per_sm = 1;
    int ahead = (inflight_per_sm + ctas_per_sm * stage_bytes - 1) / (ctas_per_sm * stage_bytes);
    int stages = ahead + 1;
    if (stages > 16) stages = 16;
    // shared memory per SM (1 KB reserved per CTA) and per CTA (1 KB left for static shared memory)
    const int64_t per_sm_budget = di.max_smem_per_sm / ctas_per_sm - 1024 - 1024;
    while (stages > 2 && ((int64_t)stages * stage_bytes + extra_bytes > per_sm_budget ||
                          (int64_t)stages * stage_bytes + extra_bytes > di.max_smem_per_block_optin - 1024))
        --stages;
    return stages < 2 ? 2 : stages;
}

}  // namespace tfk

// ---- status reporting ---------------------------------------------------------

namespace {
thread_local char g_msg[512] = "no error";
thread_local int g_inject = 0;  // cudaError_t to report instead of the next launch
}  // namespace

tfk_status tfk::fail(tfk_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

namespace {

using tfk::fail;

tfk_status ok() { return TFK_OK; }

// Launches go through the library's own (static) CUDA runtime, whose
// last-error state only this library touches: clear it before a launch so
// that the check after the launch reports that launch alone.
void clear_stale_error() { cudaGetLastError(); }

// The CUDA runtime calls on_stream_device() needs (device_scope.h).  The
// stream's device is the current one, without asking the stream, when:
// - the process sees a single device;
// - the stream is a legacy or per-thread default stream;
// - the stream is being captured into a graph: the query is refused during a
//   global-mode capture (error 900, and the capture is invalidated), and a
//   capture is made with its stream's device current, as torch.cuda.graph does.
struct CudaRuntime {
    cudaError_t stream_device(cudaStream_t s, int* dev) {
        static const int n_devices = [] {
            int n = 0;
            if (cudaGetDeviceCount(&n) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            return n;
        }();
        if (n_devices == 1 || s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread)
            return cudaGetDevice(dev);
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        const cudaError_t e = cudaStreamIsCapturing(s, &cap);
        if (e != cudaSuccess) return e;
        if (cap != cudaStreamCaptureStatusNone) return cudaGetDevice(dev);
        return cudaStreamGetDevice(s, dev);
    }
    cudaError_t current_device(int* dev) { return cudaGetDevice(dev); }
    cudaError_t set_device(int dev) { return cudaSetDevice(dev); }
};

// Runs `launch` with the stream's device current (and the caller's device
// current again afterwards).
template <class Fn>
cudaError_t on_device(void* stream, Fn&& launch) {
    CudaRuntime rt;
    return tfk::on_stream_device(rt, static_cast<cudaStream_t>(stream), launch);
}

tfk_status finish_launch(const char* op, cudaError_t err) {
    if (err != cudaSuccess)
        return fail(TFK_ERR_CUDA, "%s: CUDA error %d (%s)", op, (int)err, cudaGetErrorString(err));
    return TFK_OK;
}

// A pending injected failure replaces the launch (host-side failure testing).
bool take_injected(const char* op, tfk_status* st) {
    if (g_inject == 0) return false;
    const cudaError_t e = (cudaError_t)g_inject;
    g_inject = 0;
    *st = fail(TFK_ERR_CUDA, "%s: CUDA error %d (%s) [injected]", op, (int)e, cudaGetErrorString(e));
    return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Byte extent of `rows` rows of `width` elements at `stride` elements.
int64_t extent_bytes(int64_t rows, int64_t stride, int64_t width, int64_t es) {
    return rows <= 0 ? 0 : ((rows - 1) * stride + width) * es;
}

bool ranges_overlap(const void* a, int64_t na, const void* b, int64_t nb) {
    if (na <= 0 || nb <= 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

int64_t floor_div(int64_t a, int64_t b) {  // b > 0
    int64_t q = a / b;
    if ((a % b != 0) && (a < 0)) --q;
    return q;
}

// Do two row-strided regions (rows x width elements of size es, strides in
// elements) share any element?  Exact when the strides are equal, the usual
// case of column slices of one fused buffer; conservative otherwise.
bool regions_overlap(const void* a, int64_t sa, int64_t wa, const void* b, int64_t sb, int64_t wb,
                     int64_t rows, int64_t es) {
    if (rows <= 0 || wa <= 0 || wb <= 0) return false;
    if (!ranges_overlap(a, extent_bytes(rows, sa, wa, es), b, extent_bytes(rows, sb, wb, es))) return false;
    const int64_t dbytes = (int64_t)(reinterpret_cast<uintptr_t>(b) - reinterpret_cast<uintptr_t>(a));
    if (sa != sb || dbytes % es != 0 || sa <= 0) return true;
    const int64_t d = dbytes / es, s = sa;
    // rows i of a and i+k of b share an element iff -wb < d + k*s < wa
    int64_t k = floor_div(-wb - d, s) + 1;  // smallest k with d + k*s > -wb
    if (k < -(rows - 1)) k = -(rows - 1);
    return k <= rows - 1 && d + k * s < wa;
}

bool same_region(const void* a, int64_t sa, const void* b, int64_t sb) { return a == b && sa == sb; }

bool finite_nonneg(float v) { return std::isfinite(v) && v >= 0.0f; }

}  // namespace

extern "C" {

int tfk_abi_version(void) { return TFK_ABI_VERSION; }

const char* tfk_status_string(tfk_status s) {
    switch (s) {
        case TFK_OK: return "TFK_OK";
        case TFK_ERR_INVALID_ARGUMENT: return "TFK_ERR_INVALID_ARGUMENT";
        case TFK_ERR_MISALIGNED: return "TFK_ERR_MISALIGNED";
        case TFK_ERR_UNSUPPORTED: return "TFK_ERR_UNSUPPORTED";
        case TFK_ERR_CUDA: return "TFK_ERR_CUDA";
    }
    return "TFK_ERR_UNKNOWN";
}

const char* tfk_last_error_message(void) { return g_msg; }

tfk_status tfk_debug_fail_next_launch(int32_t cuda_error) {
    if (cuda_error < 0) return fail(TFK_ERR_INVALID_ARGUMENT, "tfk_debug_fail_next_launch: code must be >= 0");
    g_inject = cuda_error;
    return ok();
}

}  // extern "C"

namespace {

// rows are computed from x; rows [rows, padded_rows) of y are written +0.0.
// The argument checks of the RMSNorm+AdaLN entry points; *empty is set when
// the call has nothing to compute (no rows at all).
tfk_status adaln_check(const char* op, const tfk_bf16* x, int64_t x_row_stride, tfk_bf16* y,
                       int64_t y_row_stride, const float* weight, const float* shift, const float* scale,
                       const int32_t* mod_idx, int32_t n_mod, int64_t rows, int64_t padded_rows,
                       int32_t hidden, float eps, void* workspace, bool* empty) {
    *empty = false;
    if (rows < 0 || padded_rows < rows)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: need 0 <= rows (%lld) <= padded rows (%lld)", op,
                    (long long)rows, (long long)padded_rows);
    if (hidden <= 0) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: hidden = %d <= 0", op, hidden);
    if (n_mod < 1) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: n_mod = %d < 1", op, n_mod);
    if (!finite_nonneg(eps)) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: eps must be finite and >= 0", op);
    if (hidden % 8 != 0 || !tfk::rmsnorm_adaln_supported(hidden))
        return fail(TFK_ERR_UNSUPPORTED, "%s: hidden = %d (must be a multiple of 8, at most 32768)", op, hidden);
    if (x_row_stride < hidden || y_row_stride < hidden)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: row strides (%lld, %lld) must be >= hidden %d", op,
                    (long long)x_row_stride, (long long)y_row_stride, hidden);
    if (padded_rows == 0) {
        *empty = true;
        return ok();
    }
    if (!y || (rows > 0 && (!x || !weight || !shift || !scale || !mod_idx)))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: null pointer", op);
    if (x_row_stride % 8 || y_row_stride % 8)
        return fail(TFK_ERR_MISALIGNED, "%s: row strides must be multiples of 8 elements", op);
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(weight, 16) || !aligned(shift, 16) ||
        !aligned(scale, 16) || !aligned(mod_idx, 4))
        return fail(TFK_ERR_MISALIGNED, "%s: x, y, weight, shift, scale need 16-byte and mod_idx 4-byte alignment", op);
    if (!same_region(x, x_row_stride, y, y_row_stride) &&
        regions_overlap(x, x_row_stride, hidden, y, y_row_stride, hidden, padded_rows, 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: y overlaps x without being the same buffer", op);
    const int64_t ybytes = extent_bytes(padded_rows, y_row_stride, hidden, 2);
    const int64_t mbytes = (int64_t)n_mod * hidden * 4;
    if (ranges_overlap(y, ybytes, weight, (int64_t)hidden * 4) || ranges_overlap(y, ybytes, shift, mbytes) ||
        ranges_overlap(y, ybytes, scale, mbytes) || ranges_overlap(y, ybytes, mod_idx, rows * 4))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: y overlaps a parameter buffer", op);
    if (workspace) {
        const int64_t wsb = TFK_RMSNORM_WORKSPACE_BYTES;
        if (!aligned(workspace, 8)) return fail(TFK_ERR_MISALIGNED, "%s: workspace needs 8-byte alignment", op);
        if (ranges_overlap(workspace, wsb, y, ybytes) ||
            ranges_overlap(workspace, wsb, x, rows > 0 ? extent_bytes(rows, x_row_stride, hidden, 2) : 0) ||
            ranges_overlap(workspace, wsb, weight, (int64_t)hidden * 4) || ranges_overlap(workspace, wsb, shift, mbytes) ||
            ranges_overlap(workspace, wsb, scale, mbytes) || ranges_overlap(workspace, wsb, mod_idx, rows * 4))
            return fail(TFK_ERR_INVALID_ARGUMENT, "%s: workspace overlaps another argument", op);
    }
    return ok();
}

tfk_status adaln_impl(const char* op, const tfk_bf16* x, int64_t x_row_stride, tfk_bf16* y,
                      int64_t y_row_stride, const float* weight, const float* shift, const float* scale,
                      const int32_t* mod_idx, int32_t n_mod, int64_t rows, int64_t padded_rows,
                      int32_t hidden, float eps, void* workspace, void* stream) {
    bool empty = false;
    const tfk_status chk = adaln_check(op, x, x_row_stride, y, y_row_stride, weight, shift, scale, mod_idx, n_mod,
                                       rows, padded_rows, hidden, eps, workspace, &empty);
    if (chk != TFK_OK || empty) return chk;
    tfk_status st;
    if (take_injected(op, &st)) return st;
    clear_stale_error();
    tfk::AdalnArgs a{x, x_row_stride, y, y_row_stride, weight, shift, scale, mod_idx, rows, padded_rows,
                     hidden, eps, static_cast<unsigned long long*>(workspace)};
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish_launch(op, on_device(stream, [&] { return tfk::launch_rmsnorm_adaln(a, n_mod, s); }));
}

// sp_degree == 0: outputs are [padded_rows, out_row_stride] row layouts.
// sp_degree >= 1: outputs are contiguous Ulysses send buffers [sp][rows][n_heads/sp][head_dim].
tfk_status qk_impl(const char* op, const tfk_bf16* q, const tfk_bf16* k, int64_t in_row_stride,
                   tfk_bf16* q_out, tfk_bf16* k_out, int64_t out_row_stride, const float* q_weight,
                   const float* k_weight, const int32_t* positions, int64_t rows, int64_t padded_rows,
                   int32_t n_heads, int32_t head_dim, float theta, float eps, int32_t sp_degree,
                   void* stream) {
    if (rows < 0 || padded_rows < rows)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: need 0 <= rows (%lld) <= padded rows (%lld)", op,
                    (long long)rows, (long long)padded_rows);
    if (n_heads < 1 || head_dim < 1)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: n_heads = %d, head_dim = %d", op, n_heads, head_dim);
    if (!finite_nonneg(eps)) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: eps must be finite and >= 0", op);
    if (!(std::isfinite(theta) && theta > 0.0f))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: theta must be finite and > 0", op);
    if (head_dim % 16 != 0 || !tfk::qk_rope_supported(n_heads, head_dim))
        return fail(TFK_ERR_UNSUPPORTED, "%s: head_dim = %d, n_heads = %d not supported (head_dim a multiple "
                    "of 16 in [16, 512], n_heads <= 2^20)", op, head_dim, n_heads);
    if (sp_degree < 0 || (sp_degree > 0 && n_heads % sp_degree != 0))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: sp_degree %d must divide n_heads %d", op, sp_degree, n_heads);
    const int64_t width = (int64_t)n_heads * head_dim;
    if (sp_degree > 0) out_row_stride = width / sp_degree;  // row pitch inside one send block
    if (in_row_stride < width || (sp_degree == 0 && out_row_stride < width))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: row strides (%lld, %lld) must be >= n_heads*head_dim = %lld",
                    op, (long long)in_row_stride, (long long)out_row_stride, (long long)width);
    if (padded_rows == 0) return ok();
    if (!q_out || !k_out || (rows > 0 && (!q || !k || !q_weight || !k_weight || !positions)))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: null pointer", op);
    if (in_row_stride % 8 || out_row_stride % 8)
        return fail(TFK_ERR_MISALIGNED, "%s: row strides must be multiples of 8 elements", op);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(q_out, 16) || !aligned(k_out, 16) ||
        !aligned(q_weight, 16) || !aligned(k_weight, 16) || !aligned(positions, 4))
        return fail(TFK_ERR_MISALIGNED, "%s: q, k, outputs and weights need 16-byte, positions 4-byte alignment", op);
    const int64_t is = in_row_stride, os = out_row_stride;
    const int64_t orows = padded_rows;  // rows of the outputs that are written
    if (sp_degree > 0) {  // contiguous send buffers: byte ranges against everything else
        const int64_t sb = rows * width * 2, ib = extent_bytes(rows, is, width, 2);
        if (ranges_overlap(q_out, sb, k_out, sb) || ranges_overlap(q_out, sb, q, ib) ||
            ranges_overlap(q_out, sb, k, ib) || ranges_overlap(k_out, sb, q, ib) || ranges_overlap(k_out, sb, k, ib) ||
            ranges_overlap(q_out, sb, q_weight, head_dim * 4) || ranges_overlap(q_out, sb, k_weight, head_dim * 4) ||
            ranges_overlap(k_out, sb, q_weight, head_dim * 4) || ranges_overlap(k_out, sb, k_weight, head_dim * 4) ||
            ranges_overlap(q_out, sb, positions, rows * 4) || ranges_overlap(k_out, sb, positions, rows * 4))
            return fail(TFK_ERR_INVALID_ARGUMENT, "%s: a send buffer overlaps another buffer", op);
    } else {
    if (regions_overlap(q_out, os, width, k_out, os, width, orows, 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: q_out and k_out overlap", op);
    if (!same_region(q, is, q_out, os) && regions_overlap(q, is, width, q_out, os, width, orows, 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: q_out overlaps q without being the same buffer", op);
    if (!same_region(k, is, k_out, os) && regions_overlap(k, is, width, k_out, os, width, orows, 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: k_out overlaps k without being the same buffer", op);
    if (regions_overlap(q, is, width, k_out, os, width, orows, 2) ||
        regions_overlap(k, is, width, q_out, os, width, orows, 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: an output overlaps the other tensor's input", op);
    const int64_t ob = extent_bytes(orows, os, width, 2);
    const int64_t wb = (int64_t)head_dim * 4;
    if (ranges_overlap(q_out, ob, q_weight, wb) || ranges_overlap(q_out, ob, k_weight, wb) ||
        ranges_overlap(k_out, ob, q_weight, wb) || ranges_overlap(k_out, ob, k_weight, wb) ||
        ranges_overlap(q_out, ob, positions, rows * 4) || ranges_overlap(k_out, ob, positions, rows * 4))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: an output overlaps a weight or the positions", op);
    }
    tfk_status st;
    if (take_injected(op, &st)) return st;
    clear_stale_error();
    const int hpg = sp_degree > 0 ? n_heads / sp_degree : n_heads;
    const int64_t gstride = sp_degree > 0 ? rows * hpg * (int64_t)head_dim : 0;
    tfk::QkRopeArgs a{q, k, in_row_stride, q_out, k_out, out_row_stride, q_weight, k_weight,
                      positions, rows, padded_rows, hpg, gstride, n_heads, head_dim, theta, eps};
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish_launch(op, on_device(stream, [&] { return tfk::launch_qk_rmsnorm_rope(a, s); }));
}

}  // namespace

extern "C" {

tfk_status tfk_rmsnorm_adaln_indexed(const tfk_bf16* x, int64_t x_row_stride, tfk_bf16* y,
                                     int64_t y_row_stride, const float* weight, const float* shift,
                                     const float* scale, const int32_t* mod_idx, int32_t n_mod,
                                     int64_t rows, int32_t hidden, float eps, void* workspace, void* stream) {
    return adaln_impl("tfk_rmsnorm_adaln_indexed", x, x_row_stride, y, y_row_stride, weight, shift, scale,
                      mod_idx, n_mod, rows, rows, hidden, eps, workspace, stream);
}

tfk_status tfk_rmsnorm_adaln_indexed_fixed_valid(const tfk_bf16* x, int64_t x_row_stride, tfk_bf16* y,
                                                 int64_t y_row_stride, const float* weight, const float* shift,
                                                 const float* scale, const int32_t* mod_idx, int32_t n_mod,
                                                 int64_t valid_rows, int64_t padded_rows, int32_t hidden,
                                                 float eps, void* workspace, void* stream) {
    return adaln_impl("tfk_rmsnorm_adaln_indexed_fixed_valid", x, x_row_stride, y, y_row_stride, weight, shift,
                      scale, mod_idx, n_mod, valid_rows, padded_rows, hidden, eps, workspace, stream);
}

tfk_status tfk_qk_rmsnorm_rope_neox(const tfk_bf16* q, const tfk_bf16* k, int64_t in_row_stride,
                                    tfk_bf16* q_out, tfk_bf16* k_out, int64_t out_row_stride,
                                    const float* q_weight, const float* k_weight,
                                    const int32_t* positions, int64_t rows, int32_t n_heads,
                                    int32_t head_dim, float theta, float eps, void* stream) {
    return qk_impl("tfk_qk_rmsnorm_rope_neox", q, k, in_row_stride, q_out, k_out, out_row_stride, q_weight,
                   k_weight, positions, rows, rows, n_heads, head_dim, theta, eps, 0, stream);
}

tfk_status tfk_qk_rmsnorm_rope_neox_fixed_valid(const tfk_bf16* q, const tfk_bf16* k, int64_t in_row_stride,
                                                tfk_bf16* q_out, tfk_bf16* k_out, int64_t out_row_stride,
                                                const float* q_weight, const float* k_weight,
                                                const int32_t* positions, int64_t valid_rows,
                                                int64_t padded_rows, int32_t n_heads, int32_t head_dim,
                                                float theta, float eps, void* stream) {
    return qk_impl("tfk_qk_rmsnorm_rope_neox_fixed_valid", q, k, in_row_stride, q_out, k_out, out_row_stride,
                   q_weight, k_weight, positions, valid_rows, padded_rows, n_heads, head_dim, theta, eps, 0,
                   stream);
}

tfk_status tfk_qk_rmsnorm_rope_neox_ulysses(const tfk_bf16* q, const tfk_bf16* k, int64_t in_row_stride,
                                            tfk_bf16* q_send, tfk_bf16* k_send, const float* q_weight,
                                            const float* k_weight, const int32_t* positions, int64_t rows,
                                            int32_t n_heads, int32_t head_dim, int32_t sp_degree, float theta,
                                            float eps, void* stream) {
    static const char* op = "tfk_qk_rmsnorm_rope_neox_ulysses";
    if (sp_degree < 1) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: sp_degree = %d < 1", op, sp_degree);
    return qk_impl(op, q, k, in_row_stride, q_send, k_send, 0, q_weight, k_weight, positions, rows, rows,
                   n_heads, head_dim, theta, eps, sp_degree, stream);
}

static tfk_status relayout_impl(const char* op, const tfk_bf16* src, tfk_bf16* dst, int64_t row_stride,
                                int64_t rows, int32_t n_heads, int32_t head_dim, int32_t sp_degree, bool pack,
                                void* stream) {
    if (rows < 0) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: rows = %lld < 0", op, (long long)rows);
    if (n_heads < 1 || head_dim < 1 || sp_degree < 1 || n_heads % sp_degree != 0)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: n_heads %d, head_dim %d, sp_degree %d (must divide n_heads)",
                    op, n_heads, head_dim, sp_degree);
    if (head_dim % 8 != 0) return fail(TFK_ERR_UNSUPPORTED, "%s: head_dim %d is not a multiple of 8", op, head_dim);
    const int64_t width = (int64_t)n_heads * head_dim;
    if (width > (int64_t)1 << 30) return fail(TFK_ERR_UNSUPPORTED, "%s: row too wide", op);
    if (row_stride < width)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: row stride %lld < n_heads*head_dim", op, (long long)row_stride);
    if (rows == 0) return ok();
    if (!src || !dst) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: null pointer", op);
    if (row_stride % 8 || !aligned(src, 16) || !aligned(dst, 16))
        return fail(TFK_ERR_MISALIGNED, "%s: 16-byte alignment of pointers and row stride required", op);
    const void* rowbuf = pack ? (const void*)src : (const void*)dst;
    const void* grpbuf = pack ? (const void*)dst : (const void*)src;
    if (ranges_overlap(rowbuf, extent_bytes(rows, row_stride, width, 2), grpbuf, rows * width * 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: source and destination overlap", op);
    tfk_status st;
    if (take_injected(op, &st)) return st;
    clear_stale_error();
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish_launch(op, on_device(stream, [&] {
        return tfk::launch_ulysses_relayout(src, dst, row_stride, rows, n_heads, head_dim, sp_degree, pack, s);
    }));
}

tfk_status tfk_ulysses_pack(const tfk_bf16* src, int64_t src_row_stride, tfk_bf16* dst, int64_t rows,
                            int32_t n_heads, int32_t head_dim, int32_t sp_degree, void* stream) {
    return relayout_impl("tfk_ulysses_pack", src, dst, src_row_stride, rows, n_heads, head_dim, sp_degree, true,
                         stream);
}

tfk_status tfk_ulysses_unpack(const tfk_bf16* src, tfk_bf16* dst, int64_t dst_row_stride, int64_t rows,
                              int32_t n_heads, int32_t head_dim, int32_t sp_degree, void* stream) {
    return relayout_impl("tfk_ulysses_unpack", src, dst, dst_row_stride, rows, n_heads, head_dim, sp_degree, false,
                         stream);
}

tfk_status tfk_swiglu(const tfk_bf16* gate_up, int64_t in_row_stride, tfk_bf16* out,
                      int64_t out_row_stride, int64_t rows, int32_t ffn, void* stream) {
    static const char* op = "tfk_swiglu";
    if (rows < 0) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: rows = %lld < 0", op, (long long)rows);
    if (ffn <= 0) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: ffn = %d <= 0", op, ffn);
    if (ffn % 8 != 0) return fail(TFK_ERR_UNSUPPORTED, "%s: ffn = %d is not a multiple of 8", op, ffn);
    if (in_row_stride < 2LL * ffn || out_row_stride < ffn)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: row strides (%lld, %lld) must be >= (2*ffn, ffn)", op,
                    (long long)in_row_stride, (long long)out_row_stride);
    if (rows == 0) return ok();
    if (!gate_up || !out) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: null pointer", op);
    if (in_row_stride % 8 || out_row_stride % 8)
        return fail(TFK_ERR_MISALIGNED, "%s: row strides must be multiples of 8 elements", op);
    if (!aligned(gate_up, 16) || !aligned(out, 16))
        return fail(TFK_ERR_MISALIGNED, "%s: gate_up and out need 16-byte alignment", op);
    if (regions_overlap(gate_up, in_row_stride, 2LL * ffn, out, out_row_stride, ffn, rows, 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: out overlaps gate_up", op);
    tfk_status st;
    if (take_injected(op, &st)) return st;
    clear_stale_error();
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish_launch(op, on_device(stream, [&] {
        return tfk::launch_swiglu(gate_up, in_row_stride, out, out_row_stride, rows, ffn, s);
    }));
}

tfk_status tfk_valid_gather(const tfk_bf16* padded, tfk_bf16* compact, int64_t valid_rows,
                            int32_t hidden, void* stream) {
    static const char* op = "tfk_valid_gather";
    if (valid_rows < 0) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: valid_rows = %lld < 0", op, (long long)valid_rows);
    if (hidden <= 0) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: hidden = %d <= 0", op, hidden);
    if (hidden % 8 != 0) return fail(TFK_ERR_UNSUPPORTED, "%s: hidden = %d is not a multiple of 8", op, hidden);
    if (valid_rows == 0) return ok();
    if (!padded || !compact) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: null pointer", op);
    if (!aligned(padded, 16) || !aligned(compact, 16))
        return fail(TFK_ERR_MISALIGNED, "%s: buffers need 16-byte alignment", op);
    const int64_t bytes = valid_rows * hidden * 2;
    if (ranges_overlap(padded, bytes, compact, bytes))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: compact overlaps padded", op);
    tfk_status st;
    if (take_injected(op, &st)) return st;
    clear_stale_error();
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish_launch(op, on_device(stream, [&] {
        return tfk::launch_valid_gather(padded, compact, valid_rows * hidden / 8, s);
    }));
}

tfk_status tfk_zero_tail_merge(const tfk_bf16* compact, tfk_bf16* padded, int64_t valid_rows,
                               int64_t padded_rows, int32_t hidden, void* stream) {
    static const char* op = "tfk_zero_tail_merge";
    if (valid_rows < 0 || padded_rows < 0 || valid_rows > padded_rows)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: need 0 <= valid_rows (%lld) <= padded_rows (%lld)", op,
                    (long long)valid_rows, (long long)padded_rows);
    if (hidden <= 0) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: hidden = %d <= 0", op, hidden);
    if (hidden % 8 != 0) return fail(TFK_ERR_UNSUPPORTED, "%s: hidden = %d is not a multiple of 8", op, hidden);
    if (padded_rows == 0) return ok();
    if (!padded || (valid_rows > 0 && !compact)) return fail(TFK_ERR_INVALID_ARGUMENT, "%s: null pointer", op);
    if (!aligned(padded, 16) || !aligned(compact, 16))
        return fail(TFK_ERR_MISALIGNED, "%s: buffers need 16-byte alignment", op);
    if (ranges_overlap(compact, valid_rows * hidden * 2, padded, padded_rows * hidden * 2))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: compact overlaps padded", op);
    tfk_status st;
    if (take_injected(op, &st)) return st;
    clear_stale_error();
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish_launch(op, on_device(stream, [&] {
        return tfk::launch_zero_tail_merge(compact, padded, valid_rows * hidden / 8, padded_rows * hidden / 8, s);
    }));
}

}  // extern "C"

// ---- RMSNorm+AdaLN without any allocation by the caller ----------------------
//
// tfk_rmsnorm_adaln_indexed_noalloc runs the same computation as
// tfk_rmsnorm_adaln_indexed, with the scratch the warp-per-row kernel uses
// (its row counters) in an array of this library instead of a workspace from
// the caller.  The array is a file-scope device variable: every GPU that loads
// the library holds it until the process exits.  In host code its name only
// stands for it; its device address comes from cudaGetSymbolAddress, taken
// once per device with that device current and cached.  Every call uses the
// same array, so calls that may run at the same time on one GPU race on it.

namespace {

constexpr size_t kNoAllocScratchBytes = 4096;  // the array; a call needs TFK_RMSNORM_WORKSPACE_BYTES of it
static_assert(TFK_RMSNORM_WORKSPACE_BYTES <= kNoAllocScratchBytes,
              "the no-allocation scratch array is smaller than the RMSNorm workspace");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[tfk::kMaxDevicesForScratch];

// Device address of g_noalloc_scratch on the current device (set up on the
// first call for that device).
cudaError_t noalloc_scratch(void** addr) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= tfk::kMaxDevicesForScratch) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" tfk_status tfk_rmsnorm_adaln_indexed_noalloc(const tfk_bf16* x, int64_t x_row_stride, tfk_bf16* y,
                                                        int64_t y_row_stride, const float* weight,
                                                        const float* shift, const float* scale,
                                                        const int32_t* mod_idx, int32_t n_mod, int64_t rows,
                                                        int32_t hidden, float eps, void* stream) {
    static const char* op = "tfk_rmsnorm_adaln_indexed_noalloc";
    bool empty = false;
    const tfk_status chk = adaln_check(op, x, x_row_stride, y, y_row_stride, weight, shift, scale, mod_idx, n_mod,
                                       rows, rows, hidden, eps, nullptr, &empty);
    if (chk != TFK_OK || empty) return chk;
    // The scratch a call needs does not grow with its sizes, so no size can
    // exceed the array; kept as a check in case the workspace ever grows.
    if ((size_t)TFK_RMSNORM_WORKSPACE_BYTES > kNoAllocScratchBytes)
        return fail(TFK_ERR_UNSUPPORTED, "%s: needs %d bytes of scratch, more than the %zu-byte array", op,
                    TFK_RMSNORM_WORKSPACE_BYTES, kNoAllocScratchBytes);
    tfk_status st;
    if (take_injected(op, &st)) return st;
    clear_stale_error();
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish_launch(op, on_device(stream, [&]() -> cudaError_t {
        void* scratch = nullptr;
        cudaError_t err = noalloc_scratch(&scratch);
        if (err != cudaSuccess) return err;
        // The counters must start at zero: clear them on the call's stream
        // (a completed call also leaves them zero).
        if ((err = cudaMemsetAsync(scratch, 0, TFK_RMSNORM_WORKSPACE_BYTES, s)) != cudaSuccess) return err;
        tfk::AdalnArgs a{x, x_row_stride, y, y_row_stride, weight, shift, scale, mod_idx, rows, rows,
                         hidden, eps, static_cast<unsigned long long*>(scratch)};
        return tfk::launch_rmsnorm_adaln(a, n_mod, s);
    }));
}
