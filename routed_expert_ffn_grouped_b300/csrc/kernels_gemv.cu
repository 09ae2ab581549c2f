// Decode kernels: fused gate/up int4 x int8 GEMV + SwiGLU + q8(h), down GEMV, combine.
//
// Weight bytes are streamed once per call with 128-bit loads that bypass L1; each lane
// owns whole 32-element groups (16 bytes of nibbles), so a group's scale applies to
// exactly one int32 dot. Activation codes (a few KB per token) are read through L1.
#include "kernels.cuh"

namespace clb {

template <int NGL>
__global__ void __launch_bounds__(GU_WARPS * 32) k_gateup(GateUpArgs a)
{
    __shared__ int s_tok[TOK_CHUNK];
    __shared__ int s_row[TOK_CHUNK];
    __shared__ float s_h[TOK_CHUNK][GU_ROWS + 1];
    const Counters ct = *a.counters;
    const int item = blockIdx.x;
    if (item >= ct.n_items_gateup)
        return;
    const int sh_items = a.has_shared ? a.shared_ffn / G : 0;
    int slot, rb;
    if (item < sh_items) {
        slot = 0;
        rb = item;
    } else {
        const int r = item - sh_items, nrb = a.ffn / G;
        slot = (a.has_shared ? 1 : 0) + r / nrb;
        rb = r % nrb;
    }
    const Slot sd = a.slots[slot];
    const bool is_shared = sd.expert < 0;
    const colibri_expert ex = is_shared ? a.shared : a.experts[sd.expert];
    const int d = a.d, ngd = d / G, fsg = a.fmax / G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int RPW = GU_ROWS / GU_WARPS;
    const int n0 = rb * GU_ROWS + warp * RPW;

    for (int c0 = 0; c0 < sd.count; c0 += TOK_CHUNK) {
        const int nt = min(TOK_CHUNK, sd.count - c0);
        __syncthreads();
        if ((int)threadIdx.x < nt) {
            const int c = c0 + threadIdx.x;
            int t, r;
            if (is_shared) {
                t = c;
                r = a.T * a.K + c;
            } else {
                const int p = a.pairs[sd.begin + c];
                t = p / a.K;
                r = p;
            }
            s_tok[threadIdx.x] = t;
            s_row[threadIdx.x] = r;
        }
        __syncthreads();
        for (int rr = 0; rr < RPW; ++rr) {
            const int n = n0 + rr;
            const uint8_t *w1row = ex.w1 + (long)n * (d / 2);
            const uint8_t *w3row = ex.w3 + (long)n * (d / 2);
            uint4 w1v[NGL], w3v[NGL];
            float s1v[NGL], s3v[NGL];
#pragma unroll
            for (int i = 0; i < NGL; ++i) {
                const int g = lane + 32 * i;
                if (g < ngd) {
                    w1v[i] = ld_stream(w1row + g * 16);
                    w3v[i] = ld_stream(w3row + g * 16);
                    s1v[i] = __ldg(ex.s1 + (long)n * ngd + g);
                    s3v[i] = __ldg(ex.s3 + (long)n * ngd + g);
                } else {
                    w1v[i] = w3v[i] = make_uint4(0, 0, 0, 0);
                    s1v[i] = s3v[i] = 0.0f;
                }
            }
            for (int j0 = 0; j0 < nt; j0 += 4) {
                float a1[4], a3[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    a1[j] = a3[j] = 0.0f;
#pragma unroll
                for (int i = 0; i < NGL; ++i) {
                    const int g = lane + 32 * i;
                    if (g < ngd) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (j0 + j < nt) {
                                const int t = s_tok[j0 + j];
                                const int8_t *xa = a.xq_eo + (long)t * d + g * G;
                                const uint4 A0 = ld_nc(xa), A1 = ld_nc(xa + 16);
                                const int corr = __ldg(a.xc + (long)t * ngd + g);
                                const float sa = __ldg(a.xs + (long)t * ngd + g);
                                const int D1 = dot_group(w1v[i], A0, A1, corr);
                                const int D3 = dot_group(w3v[i], A0, A1, corr);
                                a1[j] = fmaf((float)D1, s1v[i] * sa, a1[j]);
                                a3[j] = fmaf((float)D3, s3v[i] * sa, a3[j]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j0 + j < nt) {
                        const float gt = warp_sum(a1[j]);
                        const float up = warp_sum(a3[j]);
                        if (lane == 0)
                            s_h[j0 + j][warp * RPW + rr] = gt / (1.0f + expf(-gt)) * up;
                    }
                }
            }
        }
        __syncthreads();
        // q8 of h over this item's 32 rows, one warp per token
        for (int j = warp; j < nt; j += GU_WARPS) {
            const float v = s_h[j][lane];
            const float amax = warp_max(fabsf(v));
            const float dd = __fdiv_rn(amax, 127.0f);
            const int q = q8_code(v, dd);
            const long r = s_row[j];
            const long hb = r * a.fmax + (long)rb * GU_ROWS;
            a.hq[hb + lane] = (int8_t)q;
            a.hq_eo[hb + eo_pos(lane)] = (int8_t)q;
            const int s = warp_sum_i(q);
            if (lane == 0) {
                a.hs[r * fsg + rb] = dd;
                a.hc[r * fsg + rb] = 8 * s;
            }
        }
    }
}

template <int NGL2>
__global__ void __launch_bounds__(DN_WARPS * 32) k_down(DownArgs a)
{
    __shared__ int s_row[TOK_CHUNK];
    const Counters ct = *a.counters;
    const int nmb = (a.d + DN_ROWS - 1) / DN_ROWS;
    const int item = blockIdx.x;
    if (item >= ct.n_items_down)
        return;
    const int slot = item / nmb, mb = item % nmb;
    const Slot sd = a.slots[slot];
    const bool is_shared = sd.expert < 0;
    const colibri_expert ex = is_shared ? a.shared : a.experts[sd.expert];
    const int f = is_shared ? a.shared_ffn : a.ffn;
    const int ngf = f / G, fsg = a.fmax / G, d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int RPW = DN_ROWS / DN_WARPS;
    constexpr int RB = 4;

    for (int c0 = 0; c0 < sd.count; c0 += TOK_CHUNK) {
        const int nt = min(TOK_CHUNK, sd.count - c0);
        __syncthreads();
        if ((int)threadIdx.x < nt) {
            const int c = c0 + threadIdx.x;
            s_row[threadIdx.x] = is_shared ? a.T * a.K + c : a.pairs[sd.begin + c];
        }
        __syncthreads();
        for (int rr0 = 0; rr0 < RPW; rr0 += RB) {
            uint4 wv[RB][NGL2];
            float sv[RB][NGL2];
#pragma unroll
            for (int b = 0; b < RB; ++b) {
                const int m = mb * DN_ROWS + warp * RPW + rr0 + b;
#pragma unroll
                for (int i = 0; i < NGL2; ++i) {
                    const int g = lane + 32 * i;
                    if (m < d && g < ngf) {
                        wv[b][i] = ld_stream(ex.w2 + (long)m * (f / 2) + g * 16);
                        sv[b][i] = __ldg(ex.s2 + (long)m * ngf + g);
                    } else {
                        wv[b][i] = make_uint4(0, 0, 0, 0);
                        sv[b][i] = 0.0f;
                    }
                }
            }
            for (int j = 0; j < nt; ++j) {
                const long r = s_row[j];
                float acc[RB];
#pragma unroll
                for (int b = 0; b < RB; ++b)
                    acc[b] = 0.0f;
#pragma unroll
                for (int i = 0; i < NGL2; ++i) {
                    const int g = lane + 32 * i;
                    if (g < ngf) {
                        const int8_t *ha = a.hq_eo + r * a.fmax + g * G;
                        const uint4 A0 = ld_nc(ha), A1 = ld_nc(ha + 16);
                        const int corr = a.hc[r * fsg + g];
                        const float sa = a.hs[r * fsg + g];
#pragma unroll
                        for (int b = 0; b < RB; ++b) {
                            const int D = dot_group(wv[b][i], A0, A1, corr);
                            acc[b] = fmaf((float)D, sv[b][i] * sa, acc[b]);
                        }
                    }
                }
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    const float v = warp_sum(acc[b]);
                    const int m = mb * DN_ROWS + warp * RPW + rr0 + b;
                    if (lane == 0 && m < d)
                        a.y[r * d + m] = v;
                }
            }
        }
    }
}

// out[t][m] = y_shared[t][m] + sum_i w[t][i] * y[t*K+i][m], fmaf chain in slot order.
__global__ void __launch_bounds__(256) k_combine(CombineArgs a)
{
    const int t = blockIdx.y;
    const int m = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (m >= a.d)
        return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.has_shared)
        acc = *reinterpret_cast<const float4 *>(a.y + ((long)a.T * a.K + t) * a.d + m);
    for (int i = 0; i < a.K; ++i) {
        const float wi = a.w[(long)t * a.K + i];
        const float4 v = *reinterpret_cast<const float4 *>(a.y + ((long)t * a.K + i) * a.d + m);
        acc.x = fmaf(wi, v.x, acc.x);
        acc.y = fmaf(wi, v.y, acc.y);
        acc.z = fmaf(wi, v.z, acc.z);
        acc.w = fmaf(wi, v.w, acc.w);
    }
    *reinterpret_cast<float4 *>(a.out + (long)t * a.d + m) = acc;
}

// Test export: one warp per row, lanes over groups, through dot_group. The plain codes
// are rearranged into even/odd words with byte permutes.
__global__ void __launch_bounds__(256) k_debug_dots(const uint8_t *w, const int8_t *qa, int rows, int cols,
                                                    int32_t *dots)
{
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows)
        return;
    const int ng = cols / G;
    for (int g = lane; g < ng; g += 32) {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(qa + g * G);
        uint32_t P[8];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            P[j] = p[j];
        for (int k = 0; k < G; ++k)
            sum += qa[g * G + k];
        uint4 A0, A1;
        A0.x = __byte_perm(P[0], P[1], 0x6420);
        A0.y = __byte_perm(P[0], P[1], 0x7531);
        A0.z = __byte_perm(P[2], P[3], 0x6420);
        A0.w = __byte_perm(P[2], P[3], 0x7531);
        A1.x = __byte_perm(P[4], P[5], 0x6420);
        A1.y = __byte_perm(P[4], P[5], 0x7531);
        A1.z = __byte_perm(P[6], P[7], 0x6420);
        A1.w = __byte_perm(P[6], P[7], 0x7531);
        const uint4 wv = *reinterpret_cast<const uint4 *>(w + (long)row * (cols / 2) + g * 16);
        dots[(long)row * ng + g] = dot_group(wv, A0, A1, 8 * sum);
    }
}

template <int NGL>
static cudaError_t gateup_n(const GateUpArgs &a, int grid, cudaStream_t s)
{
    k_gateup<NGL><<<grid, GU_WARPS * 32, 0, s>>>(a);
    return cudaGetLastError();
}

template <int NGL2>
static cudaError_t down_n(const DownArgs &a, int grid, cudaStream_t s)
{
    k_down<NGL2><<<grid, DN_WARPS * 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gateup(const GateUpArgs &a, int grid, cudaStream_t s)
{
    const int ngl = (a.d / G + 31) / 32;
    switch (ngl) {
    case 1: return gateup_n<1>(a, grid, s);
    case 2: return gateup_n<2>(a, grid, s);
    case 3: return gateup_n<3>(a, grid, s);
    case 4: return gateup_n<4>(a, grid, s);
    case 5: return gateup_n<5>(a, grid, s);
    case 6: return gateup_n<6>(a, grid, s);
    case 7: return gateup_n<7>(a, grid, s);
    case 8: return gateup_n<8>(a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_down(const DownArgs &a, int grid, cudaStream_t s)
{
    const int ngl = (a.fmax / G + 31) / 32;
    switch (ngl) {
    case 1: return down_n<1>(a, grid, s);
    case 2: return down_n<2>(a, grid, s);
    case 3: return down_n<3>(a, grid, s);
    case 4: return down_n<4>(a, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace clb
