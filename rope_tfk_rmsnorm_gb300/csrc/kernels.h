// kernels.h - internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Arguments reaching these functions have already
// been validated by the ABI layer.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tfk {

// Devices a process may use with this library's per-device caches.
constexpr int kMaxDevicesForScratch = 64;

// Attributes of the current device, read once per device and cached.
struct DeviceInfo {
    int sm_count;
    int max_smem_per_block_optin;  // bytes
    int max_smem_per_sm;           // bytes
};
cudaError_t device_info(DeviceInfo* out);

struct AdalnArgs {
    const uint16_t* x;
    int64_t x_stride;
    uint16_t* y;
    int64_t y_stride;
    const float* weight;
    const float* shift;
    const float* scale;
    const int32_t* mod_idx;
    int64_t rows;         // rows computed from x
    int64_t padded_rows;  // rows [rows, padded_rows) of y are written +0.0 (== rows: none)
    int hidden;
    float eps;
    // Optional (may be null): [0] next row to hand out, [1] CTAs finished;
    // zero before the launch, left zero by its last CTA.
    unsigned long long* sched;
};
cudaError_t launch_rmsnorm_adaln(const AdalnArgs& a, int n_mod, cudaStream_t stream);

struct QkRopeArgs {
    const uint16_t* q;
    const uint16_t* k;
    int64_t in_stride;
    uint16_t* q_out;
    uint16_t* k_out;
    int64_t out_stride;
    const float* q_weight;
    const float* k_weight;
    const int32_t* pos;
    int64_t rows;         // rows computed from q, k
    int64_t padded_rows;  // rows [rows, padded_rows) of q_out, k_out are written +0.0
    int heads_per_group;  // output head h goes to group h / heads_per_group (n_heads: one group)
    int64_t group_stride; // elements between output groups (Ulysses send layout), 0 for one group
    int n_heads;
    int head_dim;
    float theta;
    float eps;
};
cudaError_t launch_qk_rmsnorm_rope(const QkRopeArgs& a, cudaStream_t stream);

// Head <-> sequence relayout around the Ulysses all-to-all: pack copies
// [rows, stride] (n_heads heads of head_dim) into [groups][rows][n_heads/groups][head_dim];
// unpack is the inverse.
cudaError_t launch_ulysses_relayout(const uint16_t* src, uint16_t* dst, int64_t row_stride, int64_t rows,
                                   int n_heads, int head_dim, int groups, bool pack, cudaStream_t stream);

cudaError_t launch_swiglu(const uint16_t* gate_up, int64_t in_stride, uint16_t* out,
                          int64_t out_stride, int64_t rows, int ffn, cudaStream_t stream);

cudaError_t launch_valid_gather(const uint16_t* padded, uint16_t* compact, int64_t n_vec,
                                cudaStream_t stream);

cudaError_t launch_zero_tail_merge(const uint16_t* compact, uint16_t* padded, int64_t n_valid_vec,
                                   int64_t n_total_vec, cudaStream_t stream);

// Launch-shape choices, exposed so that the ABI layer can reject sizes the
// kernels do not implement before anything is enqueued.
bool rmsnorm_adaln_supported(int hidden);
bool qk_rope_supported(int n_heads, int head_dim);

// Resident CTAs per SM for `func` at this block size and dynamic shared
// memory (raising the function's dynamic shared-memory limit when needed);
// cached per device.  Returns 0 if the configuration cannot run.
int blocks_per_sm(const void* func, int threads, size_t smem_bytes);

// Depth of a cp.async staging ring (2..16 stages of `stage_bytes`) that keeps
// about `inflight_per_sm` bytes in flight per SM when `ctas_per_sm` CTAs share
// an SM, within the shared memory of the SM and of one CTA (`extra_bytes` of
// other dynamic shared memory per CTA).
#ifndef TFK_INFLIGHT_KB
#define TFK_INFLIGHT_KB 112
#endif
constexpr int kInflightPerSm = TFK_INFLIGHT_KB * 1024;
int pick_stages(int ctas_per_sm, int stage_bytes, int extra_bytes, int inflight_per_sm = kInflightPerSm);

// Programmatic dependent launch: a kernel of this library may be scheduled
// while the previous kernel on its stream drains its last CTAs.  Each kernel
// runs only setup that touches no global memory before `grid_dep_wait()`
// (common.cuh), which returns once every earlier grid of the stream has
// completed and its memory operations are visible, so stream order holds for
// any predecessor; the launch, CTA placement and that setup overlap the
// predecessor's tail.  No kernel triggers its dependents early (no
// `griddepcontrol.launch_dependents`): the implicit trigger at CTA exit
// measured best.  With an early trigger the next kernel's waiting CTAs took
// SM slots while this one still ran (per-frame chain 10% slower).
#ifndef TFK_PDL
#define TFK_PDL 1
#endif
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                          cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = TFK_PDL ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args...);
    return err != cudaSuccess ? err : cudaGetLastError();
}

// The same launch for a kernel compiled for clusters of `cluster` CTAs along x
// (the grid a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                  unsigned cluster, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = TFK_PDL ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args...);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace tfk
