// Decode on fp32 activations: the variant of the layer whose token stays in fp32, as the
// pages' one-token decode does ("Analyse approfondie", step 3 of "Guide Complet de
// Colibri"), against the same int4 group-scaled expert weights. Nothing but the weights is
// quantised: gate, up, h and y are fp32.
//
// Two kernels per layer call, each over (row block of 32 output rows, pair), a pair being
// one (token, selected expert) or (token, shared expert):
//   k_f32_gateup: h[p][n] = silu(gate_n) * up_n, gate_n = sum_g s1[n][g] * sum_k q1[n][k] x[k];
//   k_f32_down:   y[p][m] = sum_g s2[m][g] * sum_j q2[m][j] h[p][j];
// then k_combine adds the pairs' outputs with the routing weights. Lane l of a warp owns
// row l of the block and reads its 16 bytes of each 32-element group tile: the 32 lanes
// read the tile's 512 contiguous bytes. The 8 warps of a CTA split the groups; the CTA adds
// their partial sums in warp order. The activation row (x, or the pair's h) sits in shared
// memory and every lane reads the same element at a time (a broadcast).
//
// Weights are read once per pair, not once per distinct expert: a batch where several
// tokens pick one expert reads it once for each. The variant is for comparison with the
// int8-activation path at decode sizes, not a replacement for it.
#include "kernels.cuh"

namespace clb {

namespace {

constexpr int FW = 8;  // warps per CTA

// q - 8 of nibble s of word v, as an exact float: the low mantissa bits of 2^23 + n
__device__ __forceinline__ float nib(uint32_t v, int s)
{
    return __int_as_float(0x4B000000u | ((v >> s) & 15u)) - 8388616.0f;
}

// sum over the 32 elements of one group tile row (16 bytes: element 2j in the low nibble
// of byte j, 2j + 1 in the high one) times the 32 fp32 values at v (shared memory)
__device__ __forceinline__ float dot_group(uint4 w, const float *v)
{
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    const float4 *v4 = reinterpret_cast<const float4 *>(v);
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // word i holds elements 8i .. 8i+7, element 8i+e in bits 4e .. 4e+3
        const float4 a = v4[2 * i], b = v4[2 * i + 1];
        const uint32_t u = wd[i];
        acc = fmaf(nib(u, 0), a.x, acc);
        acc = fmaf(nib(u, 4), a.y, acc);
        acc = fmaf(nib(u, 8), a.z, acc);
        acc = fmaf(nib(u, 12), a.w, acc);
        acc = fmaf(nib(u, 16), b.x, acc);
        acc = fmaf(nib(u, 20), b.y, acc);
        acc = fmaf(nib(u, 24), b.z, acc);
        acc = fmaf(nib(u, 28), b.w, acc);
    }
    return acc;
}

// The pair p of a block: its expert, its token and the expert's intermediate size.
// Returns false for a routed id outside [0, E) (flagged once).
__device__ __forceinline__ bool pair_expert(const F32Args &a, int p, colibri_expert &ex, int &t, int &f)
{
    const int PK = a.T * a.K;
    if (p >= PK) {
        ex = a.shared;
        t = p - PK;
        f = a.shared_ffn;
        return true;
    }
    const int e = a.ids[p];
    t = p / a.K;
    f = a.ffn;
    if (e < 0 || e >= a.E) {
        // row block 0 exists for every pair (f >= 32), so this block always runs and the
        // flag is raised once per bad id
        if (blockIdx.x == 0 && threadIdx.x == 0)
            atomicOr(a.err, ERR_BAD_ID);
        return false;
    }
    ex = a.experts[e];
    return true;
}

// Row block rb of two matrices (or one: wb == nullptr) against v: lane's row dots, summed
// over the 32-column tiles the warp takes (g = warp, warp + FW, ...), four in flight. The
// scale of tile g is the one of its group, g >> gsh (gsh = 1 for 64-element groups).
__device__ __forceinline__ void rows_dot(const unsigned char *wa, const float *sa, const unsigned char *wb,
                                         const float *sb, const float *v, int ng, int gsh, int warp, int lane,
                                         float &acc_a, float &acc_b)
{
    wa += lane * 16;
    sa += lane;
    if (wb) {
        wb += lane * 16;
        sb += lane;
    }
    int g = warp;
    for (; g + 3 * FW < ng; g += 4 * FW) {
        uint4 qa[4], qb[4];
        float ca[4], cb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t gg = (size_t)(g + u * FW);
            qa[u] = ld_stream(wa + gg * 512);
            ca[u] = __ldg(sa + (gg >> gsh) * 32);
            if (wb) {
                qb[u] = ld_stream(wb + gg * 512);
                cb[u] = __ldg(sb + (gg >> gsh) * 32);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float *vg = v + (g + u * FW) * G;
            acc_a = fmaf(ca[u], dot_group(qa[u], vg), acc_a);
            if (wb)
                acc_b = fmaf(cb[u], dot_group(qb[u], vg), acc_b);
        }
    }
    for (; g < ng; g += FW) {
        const size_t gg = (size_t)g;
        const float *vg = v + g * G;
        acc_a = fmaf(__ldg(sa + (gg >> gsh) * 32), dot_group(ld_stream(wa + gg * 512), vg), acc_a);
        if (wb)
            acc_b = fmaf(__ldg(sb + (gg >> gsh) * 32), dot_group(ld_stream(wb + gg * 512), vg), acc_b);
    }
}

// Copies n floats (n a multiple of 4, both 16-byte aligned) into shared memory.
__device__ __forceinline__ void stage_row(float *dst, const float *src, int n)
{
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int i = threadIdx.x; i < n / 4; i += blockDim.x)
        d4[i] = __ldg(s4 + i);
}

}  // namespace

// grid (fmax / 32, pairs); dynamic shared memory: d floats
__global__ void __launch_bounds__(FW * 32) k_f32_gateup(F32Args a)
{
    extern __shared__ __align__(16) float xs[];
    __shared__ float part[2][FW][32];
    const int rb = blockIdx.x, p = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    colibri_expert ex;
    int t, f;
    const bool ok = pair_expert(a, p, ex, t, f);
    if (rb * G >= f)
        return;
    float *hrow = a.h + (size_t)p * a.fmax + (size_t)rb * G;
    if (!ok) {
        if (warp == 0)
            hrow[lane] = 0.0f;  // a bad pair contributes nothing downstream
        return;
    }
    stage_row(xs, a.x + (size_t)t * a.d, a.d);
    __syncthreads();
    const int ng = a.d / G;
    const size_t tile0 = (size_t)rb * ng, stile0 = (size_t)rb * (ng >> a.gsh);
    float gt = 0.0f, up = 0.0f;
    rows_dot(ex.w1 + tile0 * 512, ex.s1 + stile0 * 32, ex.w3 + tile0 * 512, ex.s3 + stile0 * 32, xs, ng, a.gsh, warp,
             lane, gt, up);
    part[0][warp][lane] = gt;
    part[1][warp][lane] = up;
    __syncthreads();
    if (warp == 0) {
        float gs = 0.0f, us = 0.0f;
#pragma unroll
        for (int w = 0; w < FW; ++w) {
            gs += part[0][w][lane];
            us += part[1][w][lane];
        }
        hrow[lane] = gs / (1.0f + expf(-gs)) * us;
    }
}

// grid (d / 32, pairs); dynamic shared memory: fmax floats
__global__ void __launch_bounds__(FW * 32) k_f32_down(F32Args a)
{
    extern __shared__ __align__(16) float hsm[];
    __shared__ float part[FW][32];
    const int rb = blockIdx.x, p = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    colibri_expert ex;
    int t, f;
    const bool ok = pair_expert(a, p, ex, t, f);
    float *yrow = a.y + (size_t)p * a.d + (size_t)rb * G;
    if (!ok) {
        if (warp == 0)
            yrow[lane] = 0.0f;
        return;
    }
    stage_row(hsm, a.h + (size_t)p * a.fmax, f);
    __syncthreads();
    const int ng = f / G;
    const size_t tile0 = (size_t)rb * ng, stile0 = (size_t)rb * (ng >> a.gsh);
    float acc = 0.0f, unused = 0.0f;
    rows_dot(ex.w2 + tile0 * 512, ex.s2 + stile0 * 32, nullptr, nullptr, hsm, ng, a.gsh, warp, lane, acc, unused);
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < FW; ++w)
            s += part[w][lane];
        yrow[lane] = s;
    }
}

size_t f32_smem_gateup(int d)
{
    return (size_t)d * sizeof(float);
}

size_t f32_smem_down(int fmax)
{
    return (size_t)fmax * sizeof(float);
}

}  // namespace clb
