// Combine (out = y_shared + sum_i w_i * y_i in slot order) and the group-dot test export.
// The decode GEMVs live in kernels_decode.cu (int8 activations) and kernels_f32act.cu
// (fp32 activations).
#include "kernels.cuh"

namespace clb {

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

// Test export: one thread per (row, group) of a matrix in the stored layout (row blocks of
// 32 rows, group-major), through the decode kernels' split-nibble dot. The plain codes are
// rearranged into even/odd words with byte permutes.
__global__ void __launch_bounds__(256) k_debug_dots(const uint8_t *w, const int8_t *qa, int rows, int cols,
                                                    int32_t *dots)
{
    const int ng = cols / G;
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)rows * ng)
        return;
    const int row = (int)(i / ng), g = (int)(i % ng);
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
    const size_t off = (((size_t)(row / 32) * ng + g) * 32 + row % 32) * 16;
    const uint4 wv = *reinterpret_cast<const uint4 *>(w + off);
    dots[(long)row * ng + g] = dot_split(split_nibbles(wv), A0, A1, 8 * sum);
}

}  // namespace clb
