// Prefill: grouped GEMMs of the routed experts on the tcgen05 tensor cores.
//
// The int4 weight codes and int8 activation codes are fed to kind::f16 MMAs as bf16,
// which holds every integer in [-128, 127] exactly; the products (|q_w * q_a| <= 1016)
// and their sums over one 32-element quantisation group (<= 32,512 in magnitude) are
// exact in the fp32 accumulator in tensor memory. So each K-tile is one group: two MMAs
// (K = 16 each) write a fresh accumulator, which then holds the exact int32 group dots
// D[m][n]; the epilogue threads read it back (one TMEM lane = one weight row per thread)
// and apply the group's scales, acc[m][n] += D[m][n] * s_w[m][g] * s_a[n][g], in fp32.
#include "kernels.cuh"
#include "umma.cuh"

#include <cuda_bf16.h>

namespace clb {

// ---- test export: one 128 x N x K tile of integer codes through the tensor core ------
// a int8 [128][k], b int8 [n][k] (row-major), d int32 [128][n]; n % 16 == 0, n <= 256,
// k % 16 == 0, k <= 256. One CTA of 128 threads; thread m owns row m of D.
__global__ void __launch_bounds__(128) k_debug_umma(const int8_t *a, const int8_t *b, int n, int k, int32_t *d,
                                                    int *err)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5;
    unsigned char *As = sm;
    unsigned char *Bs = sm + (size_t)UMMA_M * k * 2;
    const uint32_t ncols = n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : 256;
    if (warp == 0)
        tmem_alloc(&s_tmem, ncols);
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    // operands in the canonical layout, two codes (one bf16x2 word) at a time
    for (int i = tid; i < UMMA_M * k / 2; i += blockDim.x) {
        const int r = i / (k / 2), c = (i % (k / 2)) * 2;
        *reinterpret_cast<uint32_t *>(As + umma_off(r, c, k)) = bf16x2_of(a[r * k + c], a[r * k + c + 1]);
    }
    for (int i = tid; i < n * k / 2; i += blockDim.x) {
        const int r = i / (k / 2), c = (i % (k / 2)) * 2;
        *reinterpret_cast<uint32_t *>(Bs + umma_off(r, c, k)) = bf16x2_of(b[r * k + c], b[r * k + c + 1]);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    if (tid == 0) {
        const uint32_t idesc = umma_idesc_bf16(UMMA_M, n);
        for (int ks = 0; ks < k / UMMA_K; ++ks) {
            const uint64_t ad = umma_desc(smem_u32(As) + ks * 256, 128, k * 16);
            const uint64_t bd = umma_desc(smem_u32(Bs) + ks * 256, 128, k * 16);
            umma_bf16(tmem, ad, bd, idesc, ks > 0);
        }
        umma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < n; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                d[(long)tid * n + c0 + j] = (int32_t)v[j];
        }
    } else if (tid == 0 && err) {
        atomicOr(err, ERR_WAIT_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tmem, ncols);
}

size_t debug_umma_smem(int n, int k)
{
    return (size_t)(UMMA_M + n) * k * 2;
}

// ---- prefill grouped GEMM -------------------------------------------------------------
// Work item = (slot, 128-row tile of the weight matrix, tile of up to GT_N of the slot's
// tokens); items are ordered slot by slot, row tile by row tile, token tile innermost, so
// that CTAs working at the same time share weight tiles through L2. Persistent CTAs take
// items round robin. Warp roles in a CTA:
//   warp 0      loader: bulk-copies GS-group chunks of the weight tiles and their scales
//               (four 32-row blocks per matrix, contiguous runs) into a raw ring;
//   warp 1      MMA issuer (one thread): per group, two K = 16 MMAs per matrix into a
//               fresh TMEM accumulator (GT_TB buffers), then commits;
//   warps 2-7   converters, two per 32-column tile (64 weight rows and 32 tokens each):
//               nibbles -> bf16 A tiles (magic-number trick, k in the tensor-core order),
//               the token tile's bf16 codes -> B tile, and the tile's weight and
//               activation scales, into a converted ring;
//   warps 8-15  epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows) and columns
//               32*((w-8)/4).. (its tokens) of each group's D and accumulates
//               D * s_w * s_a in registers; at the end of an item it forms the output.
constexpr int GT_N = 64;       // tokens per item
constexpr int GT_GS = 3;       // 32-column tiles per raw (bulk-copied) stage
constexpr int GT_RR = 4;       // raw ring stages
constexpr int GT_CQ = 6;       // converted ring stages
constexpr int GT_NCONV = 2 * GT_GS;  // converter warps: two per tile of a raw chunk
constexpr int GT_EPI0 = 2 + GT_NCONV;  // first epilogue warp
constexpr int GT_NEPI = 8;     // epilogue warps: TMEM lane quarter x 32-column half
constexpr int GT_ECOL = 32;    // token columns per epilogue warp
constexpr int GT_THREADS = (GT_EPI0 + GT_NEPI) * 32;
constexpr int GT_TB = 4;       // TMEM accumulator buffers (128 columns each)

struct GemmItem {
    colibri_expert ex;
    int is_shared, mt, begin, count, n0, nt, kdim, slot;
};

// Item -> (slot, row tile, token tile). Per slot: row tiles * token tiles items.
template <int MODE>
__device__ __forceinline__ bool gemm_item(const GemmArgs &a, const int *pre, int n_slots, int item, GemmItem &it)
{
    int lo = 0, hi = n_slots;  // pre: inclusive prefix of items per slot
    if (item >= pre[n_slots - 1])
        return false;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] > item)
            hi = mid;
        else
            lo = mid + 1;
    }
    const int slot = lo;
    const int local = item - (slot ? pre[slot - 1] : 0);
    const Slot sd = a.slots[slot];
    it.slot = slot;
    it.is_shared = sd.expert < 0;
    it.ex = it.is_shared ? a.shared : a.experts[sd.expert];
    const int ntiles = (sd.count + GT_N - 1) / GT_N;
    it.mt = local / ntiles;
    const int tt = local % ntiles;
    it.n0 = tt * GT_N;
    it.nt = min(GT_N, sd.count - it.n0);
    it.begin = sd.begin;
    it.count = sd.count;
    it.kdim = MODE == MODE_GATEUP ? a.d : (it.is_shared ? a.shared_ffn : a.ffn);
    return true;
}

template <int MODE>
__device__ __forceinline__ int gemm_rows(const GemmArgs &a, int is_shared)
{
    return MODE == MODE_GATEUP ? (is_shared ? a.shared_ffn : a.ffn) : a.d;
}

// Shared memory: raw ring [GT_RR][M][ (4 blocks * GS tiles * 512) + (4 * GS * 128) ] |
// converted ring [GT_CQ][ M * 8 KB A tiles | 4 KB B tile | M * 128 sw | GT_N sa ] |
// barriers | item prefix [n_slots <= 1025].
template <int MODE>
struct GemmSmem {
    static constexpr int M = MODE == MODE_GATEUP ? 2 : 1;
    static constexpr int RAW_W = 4 * GT_GS * 512;      // one matrix's nibbles per stage
    static constexpr int RAW_S = 4 * GT_GS * 128;      // one matrix's scales per stage
    static constexpr int RAW = M * (RAW_W + RAW_S);
    static constexpr int CA = UMMA_M * 32 * 2;         // one bf16 A tile (128 x 32)
    static constexpr int CB = GT_N * 32 * 2;           // bf16 B tile (GT_N x 32)
    static constexpr int CONV = M * CA + CB + M * UMMA_M * 4 + GT_N * 4;
    static constexpr int BARS = 8 * (2 * GT_RR + 2 * GT_CQ + 2 * GT_TB) + 16;
    static constexpr int PRE = 4 * 1040;  // item prefix over at most 1025 slots
    // 64-element groups: per item parity, epilogue warp and column, the |h| max of the
    // warp's 32 rows; one mbarrier per pair of warps that share a 64-row group
    static constexpr int XCH = 2 * 4 * GT_NEPI * GT_ECOL;
    static constexpr int XBARS = 8 * GT_NEPI / 2;
    static constexpr int TOTAL = GT_RR * RAW + GT_CQ * CONV + BARS + PRE + XCH + XBARS;
};

// One group of the epilogue for one warp: per matrix m, the GT_ECOL TMEM columns of D (at
// ta + m * 64), then acc += D * (s_w * s_a), two columns per packed instruction. sw: the
// group's row scales [M][128]; sa: this warp's GT_ECOL token scales.
template <int M>
__device__ __forceinline__ void epi_accumulate(float (&acc)[M][GT_ECOL], uint32_t ta, const float *sw,
                                               const float *sa, int row)
{
    constexpr int NH = GT_ECOL / 16;
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const float swm = sw[m * UMMA_M + row];
        const float2 sw2 = make_float2(swm, swm);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            // 16 columns at a time: the registers of one load beside the accumulators
            uint32_t dv[16];
            tmem_ld16_async(ta + m * 64 + 16 * h, dv);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(sa + 16 * h + j);
                const float2 q0 = ffma2(sw2, make_float2(v.x, v.y), make_float2(0.f, 0.f));
                const float2 q1 = ffma2(sw2, make_float2(v.z, v.w), make_float2(0.f, 0.f));
                float *ac = &acc[m][16 * h + j];
                const float2 r0 = ffma2(make_float2(__uint_as_float(dv[j]), __uint_as_float(dv[j + 1])), q0,
                                        make_float2(ac[0], ac[1]));
                const float2 r1 = ffma2(make_float2(__uint_as_float(dv[j + 2]), __uint_as_float(dv[j + 3])), q1,
                                        make_float2(ac[2], ac[3]));
                ac[0] = r0.x, ac[1] = r0.y, ac[2] = r1.x, ac[3] = r1.y;
            }
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(GT_THREADS, 1) k_gemm(GemmArgs a)
{
    using L = GemmSmem<MODE>;
    constexpr int M = L::M;
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *raw = sm;
    unsigned char *conv = sm + GT_RR * L::RAW;
    uint64_t *bars = reinterpret_cast<uint64_t *>(conv + GT_CQ * L::CONV);
    uint64_t *raw_full = bars, *raw_empty = bars + GT_RR;
    uint64_t *conv_full = bars + 2 * GT_RR, *conv_empty = conv_full + GT_CQ;
    uint64_t *tm_full = conv_empty + GT_CQ, *tm_empty = tm_full + GT_TB;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tm_empty + GT_TB);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    int *pre = reinterpret_cast<int *>(reinterpret_cast<unsigned char *>(bars) + L::BARS);
    float *xch = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(pre) + L::PRE);
    uint64_t *xbar = reinterpret_cast<uint64_t *>(reinterpret_cast<unsigned char *>(xch) + L::XCH);
    const int gsh = a.group == 64 ? 1 : 0;  // 32-column tile -> group
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Counters ct = *a.counters;
    const int n_slots = ct.n_slots;

    if (warp == 0) {
        tmem_alloc(tmem_slot, 128 * GT_TB);
        if (lane == 0) {
            for (int i = 0; i < GT_RR; ++i) {
                mbar_init(&raw_full[i], 1);
                mbar_init(&raw_empty[i], GT_NCONV);
            }
            for (int i = 0; i < GT_CQ; ++i) {
                mbar_init(&conv_full[i], 2);
                mbar_init(&conv_empty[i], 1 + GT_NEPI);
            }
            for (int i = 0; i < GT_TB; ++i) {
                mbar_init(&tm_full[i], 1);
                mbar_init(&tm_empty[i], GT_NEPI);
            }
            for (int i = 0; i < GT_NEPI / 2; ++i)
                mbar_init(&xbar[i], 2);
            *abort_flag = 0;
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        // items per slot, inclusive prefix (n_slots <= 1025)
        int run = 0;
        for (int s0 = 0; s0 < n_slots; s0 += 32) {
            const int sl = s0 + lane;
            int v = 0;
            if (sl < n_slots) {
                const Slot sd = a.slots[sl];
                v = (gemm_rows<MODE>(a, sd.expert < 0) / UMMA_M) * ((sd.count + GT_N - 1) / GT_N);
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(FULL, v, o);
                if (lane >= o)
                    v += u;
            }
            if (sl < n_slots)
                pre[sl] = run + v;
            run += __shfl_sync(FULL, v, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_items = n_slots > 0 ? pre[n_slots - 1] : 0;
    auto fail = [&]() {
        atomicOr(a.err, ERR_WAIT_TIMEOUT);
        *reinterpret_cast<volatile int *>(abort_flag) = 1;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(abort_flag) != 0; };

    if (warp == 0) {
        // ---------------- loader ----------------
        if (lane == 0) {
            uint32_t st = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                GemmItem it;
                gemm_item<MODE>(a, pre, n_slots, item, it);
                const int ng = it.kdim / G;
                for (int g0 = 0; ok && g0 < ng; g0 += GT_GS, ++st) {
                    const int slot = st % GT_RR;
                    if (st >= GT_RR && !mbar_wait(&raw_empty[slot], ((st / GT_RR) - 1) & 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    if (aborted()) {
                        ok = false;
                        break;
                    }
                    const int n = min(GT_GS, ng - g0);
                    // scale tiles (one per group) of the groups the chunk's tiles belong to;
                    // with 64-element groups a chunk may start or end inside a group
                    const int ns = ((g0 + n - 1) >> gsh) - (g0 >> gsh) + 1;
                    unsigned char *dst = raw + (size_t)slot * L::RAW;
                    mbar_arrive_expect_tx(&raw_full[slot], (uint32_t)(M * 4 * (n * 512 + ns * 128)));
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const uint8_t *W = m == 0 ? (MODE == MODE_GATEUP ? it.ex.w1 : it.ex.w2) : it.ex.w3;
                        const float *S = m == 0 ? (MODE == MODE_GATEUP ? it.ex.s1 : it.ex.s2) : it.ex.s3;
                        for (int b = 0; b < 4; ++b) {
                            const size_t tile = (size_t)(it.mt * 4 + b) * ng + g0;  // 32-column tile index
                            const size_t stile = (size_t)(it.mt * 4 + b) * (ng >> gsh) + (g0 >> gsh);
                            bulk_g2s(dst + m * L::RAW_W + b * GT_GS * 512, W + tile * 512, n * 512, &raw_full[slot]);
                            bulk_g2s(dst + M * L::RAW_W + m * L::RAW_S + b * GT_GS * 128, S + stile * 32, ns * 128,
                                     &raw_full[slot]);
                        }
                    }
                }
            }
            // bounded wait for the copies issued, so that none lands after the CTA exits
            const uint32_t nwait = st < GT_RR ? st : GT_RR;
            for (uint32_t k = 1; k <= nwait; ++k)
                mbar_wait(&raw_full[(st - k) % GT_RR], ((st - k) / GT_RR) & 1);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            // one accumulator per quantisation group: a 32-column tile, or with 64-element
            // groups the two tiles of a group (four K = 16 MMAs into one buffer; the dots
            // of 64 codes, |sum| <= 65,024, stay exact in fp32)
            uint32_t cs = 0, acount = 0;  // conversion stages, accumulators
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                GemmItem it;
                gemm_item<MODE>(a, pre, n_slots, item, it);
                const int ng = it.kdim / G;
                const int nn = max(16, (it.nt + 15) & ~15);
                const uint32_t idesc = umma_idesc_bf16(UMMA_M, nn);
                for (int g = 0; g < ng; ++g, ++cs) {
                    const bool first = (g & gsh) == 0, last = (g & gsh) == gsh;
                    const int slot = cs % GT_CQ, tb = acount % GT_TB;
                    if (!mbar_wait(&conv_full[slot], (cs / GT_CQ) & 1) ||
                        (first && acount >= GT_TB && !mbar_wait(&tm_empty[tb], ((acount / GT_TB) - 1) & 1))) {
                        fail();
                        ok = false;
                        break;
                    }
                    if (aborted()) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t cb = smem_u32(conv + (size_t)slot * L::CONV);
#pragma unroll
                    for (int m = 0; m < M; ++m) {
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
                            const uint64_t ad = umma_desc(cb + m * L::CA + ks * 256, 128, 32 * 16);
                            const uint64_t bd = umma_desc(cb + M * L::CA + ks * 256, 128, 32 * 16);
                            umma_bf16(tmem + tb * 128 + m * 64, ad, bd, idesc, first ? ks : 1);
                        }
                    }
                    umma_commit(&conv_empty[slot]);
                    if (last) {
                        umma_commit(&tm_full[tb]);
                        ++acount;
                    }
                }
            }
        }
    } else if (warp < GT_EPI0) {
        // ---------------- converters (6 warps) ----------------
        // Converter warps cw and cw + 3 take tile cw of each raw chunk (GS = 3 tiles), half
        // the work each, so three tiles convert at once (a single warp's conversion is
        // latency-bound: two warps halve a tile's latency). Half hf handles row blocks
        // 2hf, 2hf + 1 of the 128-row weight tile (lane l: rows 64hf + l and 64hf + 32 + l;
        // 512 contiguous bytes per row block and group) and token 32hf + l of the token
        // tile. Nibbles become bf16 by a mask and the magic exponent 0x4300
        // (128 + nibble) minus 136, in the tensor-core k order. The token tile (bf16 codes,
        // zeros past the item's tokens) and the tokens' scales go straight from global to
        // shared memory by asynchronous copies issued first, so their L2 latency hides
        // behind the weight conversion and they hold no registers.
        const int cw = (warp - 2) % GT_GS, hf = (warp - 2) / GT_GS;
        uint32_t rs = 0, cb0 = 0;  // raw chunks seen, conversion stages of earlier chunks
        bool ok = true;
        int item = blockIdx.x, g0 = 0;
        GemmItem it;
        long arow = -1;  // activation row of this lane's token
        const int tn = lane + 32 * hf;
        auto item_rows = [&]() {
            gemm_item<MODE>(a, pre, n_slots, item, it);
            arow = -1;
            if (tn < it.nt) {
                const int cidx = it.n0 + tn;
                if (MODE == MODE_GATEUP)
                    arow = it.is_shared ? cidx : a.pairs[it.begin + cidx] / a.K;
                else
                    arow = it.is_shared ? (long)a.T * a.K + cidx : a.pairs[it.begin + cidx];
            }
        };
        if (item < n_items)
            item_rows();
        while (ok && item < n_items) {
            const int ng = it.kdim / G;
            const int rslot = rs % GT_RR;
            if (!mbar_wait(&raw_full[rslot], (rs / GT_RR) & 1)) {
                if (lane == 0)
                    fail();
                ok = false;
                break;
            }
            const unsigned char *rb = raw + (size_t)rslot * L::RAW;
            const int n = min(GT_GS, ng - g0);
            if (cw < n) {
                const uint32_t cs = cb0 + cw;
                const int slot = cs % GT_CQ;
                if (cs >= GT_CQ && !mbar_wait(&conv_empty[slot], ((cs / GT_CQ) - 1) & 1)) {
                    if (lane == 0)
                        fail();
                    ok = false;
                }
                if (ok) {
                    unsigned char *cb = conv + (size_t)slot * L::CONV;
                    const int g = g0 + cw;
                    float *sw_dst = reinterpret_cast<float *>(cb + M * L::CA + L::CB);
                    float *sa_dst = sw_dst + M * UMMA_M;
                    {
                        const bool valid = arow >= 0;
                        const uint16_t *src = valid ? a.abf + arow * a.act_stride + (long)g * G : a.abf;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            cp_async16(cb + M * L::CA + umma_off(tn, 8 * q, 32), src + 8 * q, valid ? 16 : 0);
                        cp_async4(sa_dst + tn, valid ? a.as + arow * a.act_groups + (g >> gsh) : a.as,
                                  valid ? 4 : 0);
                    }
                    const __nv_bfloat162 off136 = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
                    for (int m = 0; m < M; ++m) {
#pragma unroll
                        for (int bb = 0; bb < 2; ++bb) {
                            const int blk = 2 * hf + bb;
                            const int r = blk * 32 + lane;
                            const uint4 w =
                                *reinterpret_cast<const uint4 *>(rb + m * L::RAW_W + (blk * GT_GS + cw) * 512 + lane * 16);
                            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                // bf16 pairs (q_k, q_k+4) for k = 8j + s, s = 0..3: the mask and
                                // the magic exponent make 128 + nibble, minus 136 is q
                                uint32_t o[4];
#pragma unroll
                                for (int s2 = 0; s2 < 4; ++s2) {
                                    const uint32_t u = ((wv[j] >> (4 * s2)) & 0x000F000Fu) | 0x43004300u;
                                    const __nv_bfloat162 hv =
                                        __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&u), off136);
                                    o[s2] = *reinterpret_cast<const uint32_t *>(&hv);
                                }
                                *reinterpret_cast<uint4 *>(cb + m * L::CA + umma_off(r, 8 * j, 32)) =
                                    make_uint4(o[0], o[1], o[2], o[3]);
                            }
                            sw_dst[m * UMMA_M + r] =
                                *reinterpret_cast<const float *>(rb + M * L::RAW_W + m * L::RAW_S +
                                                                 (blk * GT_GS + (((g0 + cw) >> gsh) - (g0 >> gsh))) * 128 +
                                                                 lane * 4);
                        }
                    }
                    cp_async_wait_all();
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&conv_full[slot]);
                }
            }
            if (!ok)
                break;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&raw_empty[rslot]);
            ++rs;
            cb0 += n;
            g0 += GT_GS;
            if (g0 >= ng) {
                g0 = 0;
                item += gridDim.x;
                if (item < n_items)
                    item_rows();
            }
        }
    } else {
        // ---------------- epilogue (256 threads) ----------------
        const int e = warp - GT_EPI0;
        const int q = warp & 3, cq = e >> 2;  // TMEM lane quarter (rows), token half
        const int row = q * 32 + lane;             // row within the 128-row tile
        uint32_t cs = 0, acount = 0, xitems = 0;  // conversion stages, accumulators, items
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            GemmItem it;
            gemm_item<MODE>(a, pre, n_slots, item, it);
            const int ng = it.kdim / G;
            // a warp whose token half of the item's tile is empty skips the arithmetic
            // but keeps the barrier phases
            const bool has_cols = it.nt > cq * GT_ECOL;
            float acc[M][GT_ECOL];
#pragma unroll
            for (int m = 0; m < M; ++m)
#pragma unroll
                for (int j = 0; j < GT_ECOL; ++j)
                    acc[m][j] = 0.0f;
            // one accumulator per quantisation group (one or two conversion stages); its
            // scales are in the group's last stage
            for (int g = 0; g < ng; g += 1 + gsh, cs += 1 + gsh, ++acount) {
                const int slot = (cs + gsh) % GT_CQ, tb = acount % GT_TB;
                if (!mbar_wait(&tm_full[tb], (acount / GT_TB) & 1)) {
                    if (lane == 0)
                        fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (has_cols) {
                    const unsigned char *cb = conv + (size_t)slot * L::CONV;
                    const float *sw = reinterpret_cast<const float *>(cb + M * L::CA + L::CB);
                    const float *sa = sw + M * UMMA_M + cq * GT_ECOL;
                    const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + tb * 128 + cq * GT_ECOL;
                    epi_accumulate<M>(acc, ta, sw, sa, row);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&tm_empty[tb]);
                    for (int u = 0; u <= gsh; ++u)
                        mbar_arrive(&conv_empty[(cs + u) % GT_CQ]);
                }
            }
            if (!ok)
                break;
            // item output: columns cq * GT_ECOL + j < nt are tokens n0 + that of the slot
            const int orow = it.mt * UMMA_M + row;  // output row (h row or d row)
            if (MODE == MODE_GATEUP) {
                // h, then |h| max per column over the 32 rows of this warp; with 64-element
                // groups the two warps holding rows 64p..64p+63 (TMEM lane quarters 2p and
                // 2p + 1, same token half) exchange theirs through shared memory
#pragma unroll
                for (int j = 0; j < GT_ECOL; ++j) {
                    const float gt = acc[0][j], up = acc[M - 1][j];
                    acc[0][j] = gt / (1.0f + expf(-gt)) * up;
                    const float m = warp_max(fabsf(acc[0][j]));
                    if (gsh && lane == 0)
                        xch[((int)(xitems & 1) * GT_NEPI + e) * GT_ECOL + j] = m;
                    acc[M - 1][j] = m;
                }
                if (gsh) {
                    // warps GT_EPI0 + e pair up as (e, e ^ 1): TMEM lane quarters (2, 3) and (0, 1);
                    // one bounded mbarrier phase per item, the exchange area double-buffered
                    // by item parity (a warp writes buffer p again only after the partner
                    // has arrived for the item in between, so after it read buffer p)
                    const int partner = e ^ 1, buf = (int)(xitems & 1);
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&xbar[e >> 1]);
                    if (!mbar_wait(&xbar[e >> 1], xitems & 1)) {
                        if (lane == 0)
                            fail();
                        ok = false;
                        break;
                    }
                    ++xitems;
#pragma unroll
                    for (int j = 0; j < GT_ECOL; ++j)
                        acc[M - 1][j] = fmaxf(acc[M - 1][j], xch[(buf * GT_NEPI + partner) * GT_ECOL + j]);
                }
            }
            const int gq = a.group;
#pragma unroll
            for (int j = 0; j < GT_ECOL; ++j) {
                const int col = cq * GT_ECOL + j;
                const bool valid = col < it.nt;
                long pr = 0;
                if (valid) {
                    const int cidx = it.n0 + col;
                    pr = it.is_shared ? (long)a.T * a.K + cidx : a.pairs[it.begin + cidx];
                }
                if (MODE == MODE_GATEUP) {
                    const float h = acc[0][j], amax = acc[M - 1][j];  // |h| max of the h group
                    const float dd = __fdiv_rn(amax, 127.0f);
                    const int qv = q8_code_r(h, dd, __frcp_rn(dd));
                    if (valid) {
                        const long hb = pr * a.fmax + (long)(orow & ~31);
                        a.hbf[hb + bf16_pos(lane)] = bf16_of_int(qv);
                        if (lane == 0 && (orow % gq) < 32)
                            a.hs[pr * (a.fmax / gq) + orow / gq] = dd;
                    }
                } else if (valid) {
                    a.y[pr * a.d + orow] = acc[0][j];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128 * GT_TB);
    }
}

cudaError_t launch_gemm(int mode, const GemmArgs &a, cudaStream_t s)
{
    int dev = 0, n_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    if (mode == MODE_GATEUP) {
        const int smem = GemmSmem<MODE_GATEUP>::TOTAL;
        e = cudaFuncSetAttribute(k_gemm<MODE_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        k_gemm<MODE_GATEUP><<<n_sm, GT_THREADS, smem, s>>>(a);
    } else {
        const int smem = GemmSmem<MODE_DOWN>::TOTAL;
        e = cudaFuncSetAttribute(k_gemm<MODE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        k_gemm<MODE_DOWN><<<n_sm, GT_THREADS, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace clb
