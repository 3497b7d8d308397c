/*
 * tfk.h - C ABI of libtfk, the fused per-token elementwise hot path of a
 * joint audio-video diffusion-transformer (DiT) block, for NVIDIA GB300
 * (sm_103a).
 *
 * The operations are the fused kernels named by the TeleFuser MiniMax H3
 * pages: "perf(minimax-h3): add conservative DiT velocity reuse" (TeleFuser
 * PR #38), section 2 "Lossless optimizations from PR #37", and "[FEAT] Add
 * MiniMax H3 joint audio-video generation" (TeleFuser PR #23), "Changes
 * Made".  The pages name the fusions but print no formula; each entry point
 * below states the definition it computes.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *   never allocates, frees or synchronises, and keeps no state except a cache
 *   of device attributes.  All work is enqueued on `stream` (a cudaStream_t;
 *   NULL is the legacy default stream) and runs asynchronously.
 * - bf16 values are passed as raw 16-bit patterns (tfk_bf16).  Arithmetic is
 *   fp32 with fp32 accumulation; each output is rounded once to bf16, to
 *   nearest with ties to even.
 * - Row strides are in ELEMENTS.  bf16 row strides must be multiples of 8 and
 *   bf16 pointers 16-byte aligned (128-bit vector access); fp32 parameter
 *   pointers must be 16-byte aligned; int32 pointers 4-byte aligned.
 * - Arguments are validated on the host before anything is enqueued.  On any
 *   error the call returns a non-zero tfk_status, launches nothing and leaves
 *   every buffer untouched; tfk_last_error_message() then describes it.
 *   A zero-sized problem (rows == 0) is a valid no-op; its pointers may be NULL.
 * - Launch failures return TFK_ERR_CUDA.  Faults inside a kernel surface, as
 *   with any CUDA work, at the caller's next synchronisation.
 * - Index inputs (mod_idx) must lie in range: that is a caller precondition,
 *   not checked on the device (an out-of-range index reads out of bounds).
 */
#ifndef TFK_H
#define TFK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TFK_OK = 0,
    TFK_ERR_INVALID_ARGUMENT = 1, /* null pointer, negative size, bad overlap, bad eps/theta */
    TFK_ERR_MISALIGNED = 2,       /* pointer or stride breaks the alignment rules above */
    TFK_ERR_UNSUPPORTED = 3,      /* a size outside what the kernels implement */
    TFK_ERR_CUDA = 4              /* the CUDA runtime reported an error */
} tfk_status;

typedef uint16_t tfk_bf16; /* raw bf16 bits */

#define TFK_ABI_VERSION 2

/*
 * Bytes of the optional device workspace of the two RMSNorm+AdaLN entry
 * points (row counters for dynamic scheduling; see tfk_rmsnorm_adaln_indexed).
 */
#define TFK_RMSNORM_WORKSPACE_BYTES 2304

/* ABI version of the loaded library (TFK_ABI_VERSION at build time). */
int tfk_abi_version(void);

/* Static English name of a status code. */
const char* tfk_status_string(tfk_status status);

/* Message describing the last non-OK status returned on the calling thread. */
const char* tfk_last_error_message(void);

/*
 * Failure injection for host-side tests of callers' error handling: the next
 * entry-point call on this thread that passes argument validation returns
 * TFK_ERR_CUDA, reporting the CUDA error code `cuda_error` (> 0), instead of
 * launching.  Nothing is sent to the GPU.  cuda_error == 0 clears a pending
 * injection; a negative code returns TFK_ERR_INVALID_ARGUMENT.
 */
tfk_status tfk_debug_fail_next_launch(int32_t cuda_error);

/*
 * RMSNorm fused with indexed AdaLN modulation (TeleFuser PR #38, section 2,
 * the RMSNorm + indexed AdaLN fusion; TeleFuser PR #23, section Changes Made,
 * the indexed-modulation kernel).  For every row t, with m = mod_idx[t]:
 *
 *   inv_rms = 1 / sqrt( (1/hidden) * sum_j x[t,j]^2 + eps )
 *   y[t,j]  = bf16( x[t,j] * inv_rms * weight[j] * (1 + scale[m,j]) + shift[m,j] )
 *
 * x       [rows, x_row_stride] bf16, first `hidden` columns read.
 * y       [rows, y_row_stride] bf16, first `hidden` columns written; y == x
 *         (same pointer and stride) runs in place; any other overlap is an error.
 * weight  [hidden] fp32 norm weight.
 * shift, scale  [n_mod, hidden] fp32 modulation rows (row-major, contiguous).
 * mod_idx [rows] int32, 0 <= mod_idx[t] < n_mod (precondition).
 * hidden  multiple of 8, 8 <= hidden <= 32768.  eps >= 0.
 * workspace  optional DEVICE memory of TFK_RMSNORM_WORKSPACE_BYTES bytes,
 *         8-byte aligned, owned by the caller, or NULL.  With it, the kernels
 *         that keep the rows' modulation in shared memory hand rows to warps
 *         as they become free (a row counter in the workspace) instead of
 *         splitting the rows evenly up front, which keeps every SM busy to
 *         the end, in calls large enough for that to pay (x at least 336 KiB
 *         per SM); the output bits are the same either way.  It must be zero
 *         before its first use; every call that completes leaves it zero.
 *         Calls that may run at the same time on the GPU (other streams,
 *         graphs replayed concurrently) must not share a workspace: one per
 *         stream is enough, since calls on one stream run one after the
 *         other.  It must not overlap any other argument.
 */
tfk_status tfk_rmsnorm_adaln_indexed(const tfk_bf16* x, int64_t x_row_stride,
                                     tfk_bf16* y, int64_t y_row_stride,
                                     const float* weight, const float* shift, const float* scale,
                                     const int32_t* mod_idx, int32_t n_mod,
                                     int64_t rows, int32_t hidden, float eps,
                                     void* workspace, void* stream);

/*
 * RMSNorm + indexed AdaLN exactly as tfk_rmsnorm_adaln_indexed, for callers
 * that cannot allocate device memory.  The pages have no counterpart: this
 * is an interface of this library.
 *
 * Some callers have no way to hand the library a workspace: code that runs
 * where device allocation is not allowed or not wanted (cudaMalloc
 * synchronises the device and cannot be recorded into a stream capture, and a
 * real-time loop or a plugin running inside another runtime's stream often may
 * not call it), or that does not own an allocator at all.  This entry point
 * takes the same arguments as tfk_rmsnorm_adaln_indexed without the workspace
 * and allocates nothing: the row counters the warp-per-row kernel uses live in
 * a 4096-byte array of the library (a file-scope device variable; each GPU
 * that loads the library holds it until the process exits), of which a call
 * needs TFK_RMSNORM_WORKSPACE_BYTES whatever its sizes, so no size can exceed
 * it; sizes are limited as for tfk_rmsnorm_adaln_indexed.  Each call clears the
 * counters on its stream (cudaMemsetAsync) before its kernel.
 *
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and keeps it; make that
 *   first call before capturing a stream into a graph.
 * - Every call shares the one array, which keeps what the last call left in
 *   it: calls that may run at the same time on one GPU (on other streams)
 *   race on it and may compute wrong rows.  Issue them on one stream, or use
 *   tfk_rmsnorm_adaln_indexed with a workspace per stream.
 * Errors as for tfk_rmsnorm_adaln_indexed.
 */
tfk_status tfk_rmsnorm_adaln_indexed_noalloc(const tfk_bf16* x, int64_t x_row_stride,
                                             tfk_bf16* y, int64_t y_row_stride,
                                             const float* weight, const float* shift,
                                             const float* scale, const int32_t* mod_idx,
                                             int32_t n_mod, int64_t rows, int32_t hidden,
                                             float eps, void* stream);

/*
 * Q/K per-head RMSNorm fused with NeoX rotate-half RoPE (TeleFuser PR #38,
 * section 2, the Q/K norm + RoPE fusion; TeleFuser PR #23, section Changes
 * Made, the Q/K normalization with NeoX RoPE kernel).  For q (with q_weight)
 * and for k (with k_weight), every row t and head h, with D = head_dim:
 *
 *   n[d]       = v[t,h,d] / sqrt( (1/D) * sum_d v[t,h,d]^2 + eps ) * w[d]
 *   a_i        = pos[t] * theta^(-2i/D)                          (0 <= i < D/2)
 *   out[i]     = bf16( n[i] * cos(a_i) - n[i + D/2] * sin(a_i) )
 *   out[i+D/2] = bf16( n[i + D/2] * cos(a_i) + n[i] * sin(a_i) )
 *
 * q, k          [rows, in_row_stride] bf16, each row holds n_heads heads of
 *               head_dim values at columns [h*D, (h+1)*D); q and k may be two
 *               column slices of one fused QKV buffer.
 * q_out, k_out  [rows, out_row_stride] bf16, same head layout.  In place
 *               (q_out == q and k_out == k with equal strides) is allowed.
 * q_weight, k_weight  [head_dim] fp32, shared by every head.
 * positions     [rows] int32 token positions (any int32 value).
 * head_dim      multiple of 16, 16 <= head_dim <= 512; 1 <= n_heads <= 2^20.
 * theta > 0 (RoPE base, 10000 in the usual setting); eps >= 0.
 * The angle is reduced modulo one turn exactly enough that positions up to
 * 2^31 keep full fp32 accuracy in cos/sin.
 */
tfk_status tfk_qk_rmsnorm_rope_neox(const tfk_bf16* q, const tfk_bf16* k, int64_t in_row_stride,
                                    tfk_bf16* q_out, tfk_bf16* k_out, int64_t out_row_stride,
                                    const float* q_weight, const float* k_weight,
                                    const int32_t* positions, int64_t rows,
                                    int32_t n_heads, int32_t head_dim,
                                    float theta, float eps, void* stream);

/*
 * Fixed-valid mode of the two normalisation kernels (TeleFuser PR #38,
 * section 2: the fixed-valid and valid-only modes, and the gather / zero-tail
 * merge they make unnecessary): the kernel works directly on the padded
 * token buffer.  Rows [0, valid_rows) are computed exactly as by the entry
 * points above (reading only those rows of the inputs, mod_idx and
 * positions); rows [valid_rows, padded_rows) of the outputs are written +0.0
 * (0x0000) in the same launch and the padded tail of the inputs is never
 * read.  With this mode the valid-only pipeline needs no gather and no merge.
 *
 * Arguments as for the entry points above, with rows replaced by
 * 0 <= valid_rows <= padded_rows; outputs hold padded_rows rows; inputs need
 * only valid_rows rows.  Outputs may be the inputs (same pointer and stride);
 * any other overlap with the padded output region is an error.
 */
tfk_status tfk_rmsnorm_adaln_indexed_fixed_valid(const tfk_bf16* x, int64_t x_row_stride,
                                                 tfk_bf16* y, int64_t y_row_stride,
                                                 const float* weight, const float* shift,
                                                 const float* scale, const int32_t* mod_idx,
                                                 int32_t n_mod, int64_t valid_rows,
                                                 int64_t padded_rows, int32_t hidden, float eps,
                                                 void* workspace, void* stream);

tfk_status tfk_qk_rmsnorm_rope_neox_fixed_valid(const tfk_bf16* q, const tfk_bf16* k,
                                                int64_t in_row_stride, tfk_bf16* q_out,
                                                tfk_bf16* k_out, int64_t out_row_stride,
                                                const float* q_weight, const float* k_weight,
                                                const int32_t* positions, int64_t valid_rows,
                                                int64_t padded_rows, int32_t n_heads,
                                                int32_t head_dim, float theta, float eps,
                                                void* stream);

/*
 * Q/K RMSNorm + NeoX RoPE fused with Ulysses packing (TeleFuser PR #38,
 * section 2, the Q/K norm + RoPE fusion with the packing): the same arithmetic as
 * tfk_qk_rmsnorm_rope_neox, stored directly in the send layout of the
 * Ulysses sequence-parallel all-to-all of degree P = sp_degree:
 *
 *   q_send[p][t][j][d] = out_q[t][p*H/P + j][d]     (same for k)
 *
 * so block p (rows*H/P*D contiguous values) is what rank p receives.
 * q_send, k_send  contiguous [P, rows, n_heads/P, head_dim] bf16; must not
 *                 overlap any input.  P >= 1 and P divides n_heads; P == 1 is
 *                 the plain contiguous [rows, n_heads*head_dim] layout.
 * Other arguments and limits as for tfk_qk_rmsnorm_rope_neox.
 */
tfk_status tfk_qk_rmsnorm_rope_neox_ulysses(const tfk_bf16* q, const tfk_bf16* k, int64_t in_row_stride,
                                            tfk_bf16* q_send, tfk_bf16* k_send,
                                            const float* q_weight, const float* k_weight,
                                            const int32_t* positions, int64_t rows,
                                            int32_t n_heads, int32_t head_dim, int32_t sp_degree,
                                            float theta, float eps, void* stream);

/*
 * Ulysses head <-> sequence relayout (TeleFuser PR #23, section Changes Made,
 * the Ulysses relayout kernel), a bit-exact permutation around the all-to-all:
 *
 *   pack:    dst[p][t][j][d] = src[t][(p*H/P + j)*D + d]
 *   unpack:  dst[t][(p*H/P + j)*D + d] = src[p][t][j][d]
 *
 * The row-layout side is [rows, row_stride] bf16 (H = n_heads heads of
 * D = head_dim values per row, row_stride >= H*D, a multiple of 8); the
 * grouped side is contiguous [P, rows, H/P, D].  head_dim a multiple of 8;
 * P = sp_degree >= 1 divides n_heads.  Source and destination must not overlap.
 */
tfk_status tfk_ulysses_pack(const tfk_bf16* src, int64_t src_row_stride, tfk_bf16* dst, int64_t rows,
                            int32_t n_heads, int32_t head_dim, int32_t sp_degree, void* stream);

tfk_status tfk_ulysses_unpack(const tfk_bf16* src, tfk_bf16* dst, int64_t dst_row_stride, int64_t rows,
                              int32_t n_heads, int32_t head_dim, int32_t sp_degree, void* stream);

/*
 * SwiGLU on the FFN up-projection output (TeleFuser PR #23, section Changes
 * Made, the SwiGLU kernel):
 *
 *   out[t,j] = bf16( silu(g) * u ),  silu(g) = g / (1 + exp(-g)),
 *   g = gate_up[t, j],  u = gate_up[t, ffn + j]       (0 <= j < ffn)
 *
 * gate_up  [rows, in_row_stride] bf16, gate in columns [0, ffn), up in [ffn, 2*ffn).
 * out      [rows, out_row_stride] bf16, first ffn columns written; must not
 *          overlap gate_up.
 * ffn      multiple of 8, >= 8.
 */
tfk_status tfk_swiglu(const tfk_bf16* gate_up, int64_t in_row_stride,
                      tfk_bf16* out, int64_t out_row_stride,
                      int64_t rows, int32_t ffn, void* stream);

/*
 * Valid-only gather (TeleFuser PR #38, section 2, the gather fused with the
 * zero-tail merge): copy the valid prefix of a padded token buffer into a
 * compact buffer, bit for bit.
 *
 *   compact[i, :] = padded[i, :]     for 0 <= i < valid_rows
 *
 * padded   [>= valid_rows, hidden] bf16, contiguous rows.
 * compact  [valid_rows, hidden] bf16, contiguous; must not overlap padded.
 * hidden   multiple of 8.  A buffer made of several padded segments (video
 *          then audio) is handled by one call per segment with offset pointers.
 */
tfk_status tfk_valid_gather(const tfk_bf16* padded, tfk_bf16* compact,
                            int64_t valid_rows, int32_t hidden, void* stream);

/*
 * Zero-tail merge, the write-back half of the same fusion: one launch writes
 * the compact rows back and fills the padded tail with +0.0 (bits 0x0000).
 *
 *   padded[i, :] = compact[i, :]     for 0 <= i < valid_rows
 *   padded[i, :] = +0.0              for valid_rows <= i < padded_rows
 *
 * compact  [valid_rows, hidden] bf16, contiguous.
 * padded   [padded_rows, hidden] bf16, contiguous; must not overlap compact.
 * 0 <= valid_rows <= padded_rows; valid_rows == 0 zeroes the whole buffer.
 */
tfk_status tfk_zero_tail_merge(const tfk_bf16* compact, tfk_bf16* padded,
                               int64_t valid_rows, int64_t padded_rows, int32_t hidden,
                               void* stream);

/*
 * Conservative DiT velocity-cache schedule ("perf(minimax-h3): add
 * conservative DiT velocity reuse", TeleFuser PR #38, section 3).  Host-only:
 * no GPU work, no stream.
 *
 * reuse[i] = 1 when step i (0-based, progress i/num_steps) may skip the DiT
 * call and reuse the previous video/audio velocity: the progress lies in
 * [start_ratio, end_ratio), a velocity was computed on an earlier step, and
 * fewer than min(max_consecutive_reuse, refresh_interval - 1) steps in a row
 * have reused it since the last DiT call.  reuse[i] = 0 means the DiT runs.
 * The page's defaults are 0.2, 0.8, 2, 1; over 49 steps they give 15 hits
 * and 34 DiT calls.
 *
 * reuse      [num_steps] HOST array written by the call (may be NULL if num_steps == 0).
 * num_reuse  optional HOST pointer receiving the number of hits.
 * Errors: TFK_ERR_INVALID_ARGUMENT for num_steps < 0, refresh_interval < 1,
 * max_consecutive_reuse < 0, ratios outside 0 <= start <= end <= 1, or a NULL reuse.
 */
tfk_status tfk_velocity_cache_schedule(int32_t num_steps, double start_ratio, double end_ratio,
                                       int32_t refresh_interval, int32_t max_consecutive_reuse,
                                       uint8_t* reuse, int32_t* num_reuse);

#ifdef __cplusplus
}
#endif

#endif /* TFK_H */
