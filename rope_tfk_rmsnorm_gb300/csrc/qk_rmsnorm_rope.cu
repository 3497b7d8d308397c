// qk_rmsnorm_rope.cu - Q/K per-head RMSNorm fused with NeoX rotate-half RoPE.
//
// For q (weight wq) and k (weight wk), each token t and head h (D = head_dim):
//   n[d]       = v[d] * rsqrt(mean_d v^2 + eps) * w[d]
//   a_i        = pos[t] * theta^(-2i/D),  i < D/2
//   out[i]     = n[i] cos a_i - n[i+D/2] sin a_i
//   out[i+D/2] = n[i+D/2] cos a_i + n[i] sin a_i
// ("Fuse Q/K RMSNorm, RoPE, and Ulysses packing", TeleFuser PR #38 section 2;
// "Q/K normalization plus NeoX RoPE", TeleFuser PR #23 "Changes Made").
//
// Design (HBM-bound: 4 bytes per q/k element read + written, plus 4 B/token):
// - Persistent CTAs over contiguous token runs.  A head is served by G lanes
//   (G = D/16 rounded up to a power of two); lane l holds the 8-element
//   vector l of the first half and vector l of the second half, so every
//   rotate-half pair sits in one thread and needs no shuffle.  The per-head
//   sum of squares is a G-lane shuffle reduction.
// - q/k head rows are staged through a shared-memory ring with cp.async,
//   stages-1 tokens ahead; each thread reads back only its own slots.
// - cos/sin of the D/2 angles of a token are computed once per CTA per token
//   into a double-buffered shared table (the next token's table is built
//   while the current token is finished), one barrier per token.
// - The output can go straight into the Ulysses all-to-all send layout
//   [groups][rows][heads/groups][D] ("Fuse Q/K RMSNorm, RoPE, and Ulysses
//   packing", TeleFuser PR #38 section 2): only the store address changes.
// - Angles are reduced exactly in integer arithmetic: theta^(-2i/D)/(2 pi) is
//   held as a 64-bit fixed-point fraction of a turn F_i (computed once per
//   CTA in fp64), pos * F_i mod 2^64 is the angle's fraction of a turn, and
//   its top 32 bits give an fp32 angle in [-pi, pi) for sincosf.  The error
//   of the reduced angle is below 2^-40 turn for any int32 position, so no
//   fp64 work is needed per token (fp64 throughput on GB300 is low).
#include "common.cuh"
#include "kernels.h"

namespace tfk {
namespace {

constexpr int kMaxThreads = 512;

__device__ __forceinline__ float2 rope_cos_sin(int32_t pos, uint64_t turn_fraction) {
    const uint64_t a = (uint64_t)(int64_t)pos * turn_fraction;        // mod 2^64 = mod one turn
    const int32_t top = (int32_t)(uint32_t)(a >> 32);                   // [-2^31, 2^31) -> [-pi, pi)
    const float angle = (float)top * 1.46291807926715968e-9f;           // 2 pi / 2^32
    float s, c;
    sincosf(angle, &s, &c);
    return make_float2(c, s);
}

template <int HPT>
__global__ void __launch_bounds__(kMaxThreads) qk_rope_kernel(const QkRopeArgs a, const int lanes_per_head,
                                                              const int stages) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int nt = blockDim.x;
    const int tid = threadIdx.x;
    const int D = a.head_dim;
    const int half = D >> 1;
    const int L = D >> 4;                 // lanes holding data per head
    const int G = lanes_per_head;         // power of two >= L
    const int slots = 2 * a.n_heads;      // q heads then k heads
    const int heads_per_pass = nt / G;
    const float inv_d = 1.0f / (float)D;

    Vec8* ring = reinterpret_cast<Vec8*>(smem_raw);                   // [stages][HPT][2][nt]
    const int stage_vecs = HPT * 2 * nt;
    uint64_t* ftab = reinterpret_cast<uint64_t*>(ring + (int64_t)stages * stage_vecs);  // [half]
    float2* cs = reinterpret_cast<float2*>(ftab + half);              // [2][half]

    const int64_t r0 = a.rows * (int64_t)blockIdx.x / gridDim.x;
    const int64_t r1 = a.rows * (int64_t)(blockIdx.x + 1) / gridDim.x;
    const int nrows = (int)(r1 - r0);

    // Fixed-point turn fractions of the D/2 frequencies.  Thread tid owns the
    // entries i = tid (mod nt) and is the only one to read them back.
    for (int i = tid; i < half; i += nt) {
        const double f = pow((double)a.theta, -2.0 * (double)i / (double)D);
        double turns = f * 0.15915494309189533577;  // 1 / (2 pi)
        turns -= floor(turns);
        ftab[i] = __double2ull_rz(turns * 18446744073709551616.0);  // * 2^64
    }

    const int lane = tid % G;
    int slot[HPT];
    bool active[HPT];
    const uint16_t* src0[HPT];
    uint16_t* dst0[HPT];
    float wa[HPT][8], wb[HPT][8];
#pragma unroll
    for (int j = 0; j < HPT; ++j) {
        slot[j] = tid / G + j * heads_per_pass;
        active[j] = slot[j] < slots && lane < L;
        const bool is_q = slot[j] < a.n_heads;
        const int h = is_q ? slot[j] : slot[j] - a.n_heads;
        const int64_t col = (int64_t)h * D + lane * 8;
        src0[j] = (is_q ? a.q : a.k) + col;
        // output head h: group h / hpg at group_stride, head h % hpg inside the group's row
        const int grp = h / a.heads_per_group;
        dst0[j] = (is_q ? a.q_out : a.k_out) + (int64_t)grp * a.group_stride +
                  (int64_t)(h - grp * a.heads_per_group) * D + lane * 8;
        const float* wsrc = is_q ? a.q_weight : a.k_weight;
        if (active[j]) {
            const float4 x0 = ld_f4(wsrc + lane * 8), x1 = ld_f4(wsrc + lane * 8 + 4);
            const float4 y0 = ld_f4(wsrc + half + lane * 8), y1 = ld_f4(wsrc + half + lane * 8 + 4);
            wa[j][0] = x0.x; wa[j][1] = x0.y; wa[j][2] = x0.z; wa[j][3] = x0.w;
            wa[j][4] = x1.x; wa[j][5] = x1.y; wa[j][6] = x1.z; wa[j][7] = x1.w;
            wb[j][0] = y0.x; wb[j][1] = y0.y; wb[j][2] = y0.z; wb[j][3] = y0.w;
            wb[j][4] = y1.x; wb[j][5] = y1.y; wb[j][6] = y1.z; wb[j][7] = y1.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) { wa[j][e] = 0.f; wb[j][e] = 0.f; }
        }
    }

    auto issue = [&](int row_in_run, int stage) {
        const int64_t roff_in = (r0 + row_in_run) * a.in_stride;
        Vec8* st = ring + (int64_t)stage * stage_vecs;
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
            if (active[j]) {
                cp_async16(st + (j * 2 + 0) * nt + tid, src0[j] + roff_in);
                cp_async16(st + (j * 2 + 1) * nt + tid, src0[j] + roff_in + half);
            }
        }
    };

    if (nrows > 0) {  // uniform over the CTA
    for (int s = 0; s < stages - 1; ++s) {
        if (s < nrows) issue(s, s);
        cp_async_commit();
    }
    {   // cos/sin table of the first token
        const int32_t p = __ldg(a.pos + r0);
        for (int i = tid; i < half; i += nt) cs[i] = rope_cos_sin(p, ftab[i]);
    }

    for (int it = 0; it < nrows; ++it) {
        const int64_t r = r0 + it;
        const int ahead = it + stages - 1;
        if (ahead < nrows) issue(ahead, ahead % stages);
        cp_async_commit();
        cp_async_wait_dyn(stages - 1);
        __syncthreads();  // publishes cs[it & 1]

        const Vec8* st = ring + (int64_t)(it % stages) * stage_vecs;
        const float2* tab = cs + (it & 1) * half + lane * 8;
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
            float va[8], vb[8];
            float ss = 0.f;
            if (active[j]) {
                unpack8(ld_smem_vec(st + (j * 2 + 0) * nt + tid), va);
                unpack8(ld_smem_vec(st + (j * 2 + 1) * nt + tid), vb);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(va[e], va[e], fmaf(vb[e], vb[e], ss));
            }
            for (int o = G >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
            if (active[j]) {
                const float inv_rms = rsqrtf(ss * inv_d + a.eps);
                float oa[8], ob[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 c = tab[e];
                    const float na = va[e] * inv_rms * wa[j][e];
                    const float nb = vb[e] * inv_rms * wb[j][e];
                    oa[e] = fmaf(na, c.x, -nb * c.y);
                    ob[e] = fmaf(nb, c.x, na * c.y);
                }
                const int64_t roff = r * a.out_stride;
                st_vec(dst0[j] + roff, pack8(oa));
                st_vec(dst0[j] + roff + half, pack8(ob));
            }
        }

        if (it + 1 < nrows) {  // next token's table, into the other buffer
            const int32_t p = __ldg(a.pos + r + 1);
            float2* nxt = cs + ((it + 1) & 1) * half;
            for (int i = tid; i < half; i += nt) nxt[i] = rope_cos_sin(p, ftab[i]);
        }
    }
    cp_async_wait<0>();
    }  // nrows > 0

    // Fixed-valid mode: this CTA's share of the padded tail rows of q_out and
    // k_out is written +0.0 in the same launch (the input tail is never read).
    const int64_t tail = a.padded_rows - a.rows;
    if (tail > 0) {
        const int64_t z0 = a.rows + tail * (int64_t)blockIdx.x / gridDim.x;
        const int64_t z1 = a.rows + tail * (int64_t)(blockIdx.x + 1) / gridDim.x;
        Vec8 zero;
        zero.w[0] = zero.w[1] = zero.w[2] = zero.w[3] = 0u;
        for (int64_t r = z0; r < z1; ++r) {
            const int64_t roff = r * a.out_stride;
#pragma unroll
            for (int j = 0; j < HPT; ++j) {
                if (active[j]) {
                    st_vec(dst0[j] + roff, zero);
                    st_vec(dst0[j] + roff + half, zero);
                }
            }
        }
    }
}

struct Shape {
    int hpt, threads, lanes;
};

bool choose_shape(int n_heads, int head_dim, Shape* s) {
    if (head_dim < 16 || head_dim > 512 || head_dim % 16 != 0 || n_heads < 1) return false;
    int L = head_dim / 16, G = 1;
    while (G < L) G <<= 1;
    const int64_t slots = 2LL * n_heads;
    for (int hpt = 1; hpt <= 4; hpt *= 2) {
        const int64_t t = (slots + hpt - 1) / hpt * G;
        const int64_t threads = (t + 31) / 32 * 32;
        if (threads <= kMaxThreads) {
            s->hpt = hpt;
            s->threads = (int)threads;
            s->lanes = G;
            return true;
        }
    }
    return false;
}

template <int HPT>
cudaError_t launch_h(const QkRopeArgs& a, const Shape& s, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int stage_bytes = HPT * 2 * s.threads * 16;
    const int table_bytes = (a.head_dim / 2) * (8 + 2 * 8);
    const void* fn = reinterpret_cast<const void*>(&qk_rope_kernel<HPT>);
    const int by_regs = blocks_per_sm(fn, s.threads, table_bytes);
    if (by_regs <= 0) return cudaErrorInvalidConfiguration;
    const int stages = pick_stages(by_regs >= 2 ? 2 : 1, stage_bytes, table_bytes);
    const size_t smem = (size_t)stages * stage_bytes + table_bytes;
    const int per_sm = blocks_per_sm(fn, s.threads, smem);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)per_sm * di.sm_count;
    const int64_t work = a.rows > a.padded_rows - a.rows ? a.rows : a.padded_rows - a.rows;
    if (grid > work) grid = work;
    if (grid < 1) return cudaSuccess;
    qk_rope_kernel<HPT><<<(unsigned)grid, s.threads, smem, stream>>>(a, s.lanes, stages);
    return cudaGetLastError();
}

}  // namespace

bool qk_rope_supported(int n_heads, int head_dim) {
    Shape s;
    return choose_shape(n_heads, head_dim, &s);
}

cudaError_t launch_qk_rmsnorm_rope(const QkRopeArgs& a, cudaStream_t stream) {
    Shape s;
    if (!choose_shape(a.n_heads, a.head_dim, &s)) return cudaErrorInvalidValue;
    switch (s.hpt) {
        case 1: return launch_h<1>(a, s, stream);
        case 2: return launch_h<2>(a, s, stream);
        default: return launch_h<4>(a, s, stream);
    }
}

}  // namespace tfk
