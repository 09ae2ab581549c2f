// Decode GEMVs: fused gate/up + SwiGLU + q8(h), and down.
//
// Expert matrices are stored in row blocks of 32 rows, group-major inside a block: the 16
// bytes of one 32-column group of the block's 32 rows lie together (512 bytes), and the
// whole block is one contiguous run. A work item is one row block of one expert slot (32
// rows of W1 and W3 for gate/up: one group of h; 32 rows of W2 for down).
//
// One persistent CTA per SM takes a contiguous range of items. Its producer warp streams
// each item's run through a ring of NS shared-memory stages with 1-D bulk copies (a stage
// is SG group tiles of every matrix plus their scales, a few large copies), completion
// counted on a "full" mbarrier per stage. So the bytes in flight per SM are set by the
// ring (well over 100 KB), not by registers. The consumer warps split each stage's
// groups; lane l owns row l of the block and reads its 16 bytes of a group tile from
// shared memory (512 contiguous bytes per warp, no bank conflicts), so a lane accumulates
// whole row dots over its groups in registers without any cross-lane reduction. At the
// end of an item the consumers' partial sums meet in shared memory in a fixed order.
//
// The activation codes (even/odd word order, with scales and +8 corrections) of the
// item's tokens are staged in shared memory when the slot (or token chunk) changes and
// read as broadcasts. A slot with more tokens than a chunk holds is processed chunk by
// chunk, its weights streamed once per chunk.
#include "kernels.cuh"

namespace clb {

namespace {

struct DecItem {
    colibri_expert ex;
    int slot, is_shared, rb, begin, count, kdim;
};

template <int MODE>
__device__ __forceinline__ DecItem item_info(const DecodeArgs &a, int item)
{
    DecItem it;
    if (MODE == MODE_GATEUP) {
        const int sh_items = a.has_shared ? a.shared_ffn / G : 0;
        if (item < sh_items) {
            it.slot = 0;
            it.rb = item;
        } else {
            const int r = item - sh_items, nrb = a.ffn / G;
            it.slot = (a.has_shared ? 1 : 0) + r / nrb;
            it.rb = r % nrb;
        }
    } else {
        const int nmb = a.d / G;
        it.slot = item / nmb;
        it.rb = item % nmb;
    }
    const Slot sd = a.slots[it.slot];
    it.is_shared = sd.expert < 0;
    it.ex = it.is_shared ? a.shared : a.experts[sd.expert];
    it.begin = sd.begin;
    it.count = sd.count;
    it.kdim = MODE == MODE_GATEUP ? a.d : (it.is_shared ? a.shared_ffn : a.ffn);
    return it;
}

// Dynamic shared memory: ring [NS][stage] | full [NS] | empty [NS] | abort flag (16 B) |
// activation codes [TCH][Kmax] | scales [TCH][Kmax/32] | corrections [TCH][Kmax/32] |
// partial sums [2][NC][M][TCH][32] | activation rows [TCH] | output rows [TCH].
struct RingSmem {
    unsigned char *ring;
    uint64_t *full, *empty;
    int *abort_flag;
    int8_t *codes;
    float *sc;
    int *corr;
    float *part;
    int *arow, *orow;
};

__device__ __forceinline__ RingSmem carve(unsigned char *sm, const DecodeArgs &a, int nc, int m, int tch)
{
    RingSmem s;
    const int ngm = a.kmax / G;
    s.ring = sm;
    s.full = reinterpret_cast<uint64_t *>(sm + (size_t)a.ring * a.stage_bytes);
    s.empty = s.full + a.ring;
    s.abort_flag = reinterpret_cast<int *>(s.empty + a.ring);
    s.codes = reinterpret_cast<int8_t *>(s.abort_flag + 4);
    s.sc = reinterpret_cast<float *>(s.codes + (size_t)tch * a.kmax);
    s.corr = reinterpret_cast<int *>(s.sc + (size_t)tch * ngm);
    s.part = reinterpret_cast<float *>(s.corr + (size_t)tch * ngm);
    s.arow = reinterpret_cast<int *>(s.part + (size_t)2 * nc * m * tch * 32);
    s.orow = s.arow + tch;
    return s;
}

}  // namespace

// Bytes of dynamic shared memory besides the ring (host side mirror of carve()).
static size_t ring_fixed_bytes(int kmax, int nc, int m, int tch, int ns)
{
    const size_t ngm = kmax / G;
    return 16 * (size_t)ns + 16 + (size_t)tch * kmax + 8 * (size_t)tch * ngm +
           4 * (size_t)2 * nc * m * tch * 32 + 8 * (size_t)tch;
}

// MODE_GATEUP: M = 2 matrices (W1, W3), output h codes; MODE_DOWN: M = 1 (W2), output y.
// NC consumer warps + 1 producer warp; TCH tokens per chunk; a stage holds SG = NC * GPW
// groups and consumer warp w takes groups w, w + NC, ... of it.
template <int MODE, int NC, int TCH, int GPW>
__global__ void __launch_bounds__((NC + 1) * 32, 1) k_ring(DecodeArgs a)
{
    constexpr int M = MODE == MODE_GATEUP ? 2 : 1;
    constexpr int SG = NC * GPW;
    extern __shared__ __align__(128) unsigned char sm[];
    const RingSmem s = carve(sm, a, NC, M, TCH);
    const int NS = a.ring;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = MODE == MODE_GATEUP ? a.counters->n_items_gateup : a.counters->n_items_down;
    const int i0 = (int)((long)blockIdx.x * n_items / gridDim.x);
    const int i1 = (int)((long)(blockIdx.x + 1) * n_items / gridDim.x);
    // stage layout: M group-tile runs of SG*512 bytes, then M scale runs of SG*128 bytes
    constexpr int scale_off = M * SG * 512;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], NC);
        }
        *s.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NC) {
        // ---------------- producer ----------------
        if (lane != 0)
            return;
        uint32_t st = 0;
        auto drain = [&]() {  // bounded wait for the copies issued, before the CTA exits
            const uint32_t n = st < (uint32_t)NS ? st : (uint32_t)NS;
            for (uint32_t k = 1; k <= n; ++k) {
                const uint32_t q = st - k;
                mbar_wait(&s.full[q % NS], (q / NS) & 1);
            }
        };
        for (int item = i0; item < i1; ++item) {
            const DecItem it = item_info<MODE>(a, item);
            const int ng = it.kdim / G, spi = (ng + SG - 1) / SG;
            const int nch = (it.count + TCH - 1) / TCH;
            const size_t blk = (size_t)it.rb * ng;  // first group tile of the row block
            for (int ch = 0; ch < nch; ++ch) {
                for (int k = 0; k < spi; ++k, ++st) {
                    const int slot = st % NS;
                    if (st >= (uint32_t)NS && !mbar_wait(&s.empty[slot], ((st / NS) - 1) & 1)) {
                        atomicOr(a.err, ERR_WAIT_TIMEOUT);
                        *reinterpret_cast<volatile int *>(s.abort_flag) = 1;
                        drain();
                        return;
                    }
                    if (*reinterpret_cast<volatile int *>(s.abort_flag)) {
                        drain();
                        return;
                    }
                    const int g0 = k * SG, n = min(SG, ng - g0);
                    unsigned char *dst = s.ring + (size_t)slot * a.stage_bytes;
                    mbar_arrive_expect_tx(&s.full[slot], (uint32_t)(M * n * (512 + 128)));
                    if (MODE == MODE_GATEUP) {
                        bulk_g2s(dst, it.ex.w1 + (blk + g0) * 512, n * 512, &s.full[slot]);
                        bulk_g2s(dst + SG * 512, it.ex.w3 + (blk + g0) * 512, n * 512, &s.full[slot]);
                        bulk_g2s(dst + scale_off, it.ex.s1 + (blk + g0) * 32, n * 128, &s.full[slot]);
                        bulk_g2s(dst + scale_off + SG * 128, it.ex.s3 + (blk + g0) * 32, n * 128, &s.full[slot]);
                    } else {
                        bulk_g2s(dst, it.ex.w2 + (blk + g0) * 512, n * 512, &s.full[slot]);
                        bulk_g2s(dst + scale_off, it.ex.s2 + (blk + g0) * 32, n * 128, &s.full[slot]);
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    constexpr int NT = NC * 32;
    uint32_t st = 0;
    int buf = 0;
    int staged_slot = -1, staged_ch = -1;
    for (int item = i0; item < i1; ++item) {
        const DecItem it = item_info<MODE>(a, item);
        const int K = it.kdim, ng = K / G, spi = (ng + SG - 1) / SG;
        const int nch = (it.count + TCH - 1) / TCH;
        for (int ch = 0; ch < nch; ++ch) {
            const int c0 = ch * TCH, nt = min(TCH, it.count - c0);
            if (it.slot != staged_slot || ch != staged_ch) {
                // stage this chunk's activation rows (all consumers)
                named_sync(1, NT);
                if ((int)threadIdx.x < nt) {
                    const int c = c0 + threadIdx.x;
                    const int p = it.is_shared ? a.T * a.K + c : a.pairs[it.begin + c];
                    s.arow[threadIdx.x] = MODE == MODE_GATEUP ? (it.is_shared ? c : p / a.K) : p;
                    s.orow[threadIdx.x] = p;
                }
                named_sync(1, NT);
                const int v16 = K / 16;
                for (int i = threadIdx.x; i < nt * v16; i += NT) {
                    const int tt = i / v16, o = i % v16;
                    const uint4 v = ld_nc(a.aq_eo + (long)s.arow[tt] * a.act_stride + o * 16);
                    reinterpret_cast<uint4 *>(s.codes + (size_t)tt * K)[o] = v;
                }
                for (int i = threadIdx.x; i < nt * ng; i += NT) {
                    const int tt = i / ng, g = i % ng;
                    s.sc[i] = a.as[(long)s.arow[tt] * a.act_groups + g];
                    s.corr[i] = a.ac[(long)s.arow[tt] * a.act_groups + g];
                }
                named_sync(1, NT);
                staged_slot = it.slot;
                staged_ch = ch;
            }
            float acc[M][TCH];
#pragma unroll
            for (int m = 0; m < M; ++m)
#pragma unroll
                for (int t = 0; t < TCH; ++t)
                    acc[m][t] = 0.0f;
            bool aborted = false;
            for (int k = 0; k < spi; ++k, ++st) {
                const int slot = st % NS;
                if (!mbar_wait(&s.full[slot], (st / NS) & 1)) {
                    if (lane == 0)
                        atomicOr(a.err, ERR_WAIT_TIMEOUT);
                    *reinterpret_cast<volatile int *>(s.abort_flag) = 1;
                    aborted = true;
                    break;
                }
                const unsigned char *stg = s.ring + (size_t)slot * a.stage_bytes;
                const int g0 = k * SG, n = min(SG, ng - g0);
#pragma unroll
                for (int u = 0; u < GPW; ++u) {
                    const int j = warp + u * NC;
                    if (j < n) {
                        const int g = g0 + j;
                        NibbleSplit ns[M];
                        float sw[M];
#pragma unroll
                        for (int m = 0; m < M; ++m) {
                            ns[m] = split_nibbles(*reinterpret_cast<const uint4 *>(stg + (m * SG + j) * 512 + lane * 16));
                            sw[m] = *reinterpret_cast<const float *>(stg + scale_off + (m * SG + j) * 128 + lane * 4);
                        }
#pragma unroll
                        for (int t = 0; t < TCH; ++t) {
                            if (t < nt) {
                                const uint4 *xa = reinterpret_cast<const uint4 *>(s.codes + (size_t)t * K + g * G);
                                const uint4 A0 = xa[0], A1 = xa[1];
                                const int corr = s.corr[t * ng + g];
                                const float sa = s.sc[t * ng + g];
#pragma unroll
                                for (int m = 0; m < M; ++m) {
                                    const int D = dot_split(ns[m], A0, A1, corr);
                                    acc[m][t] = fmaf((float)D, sw[m] * sa, acc[m][t]);
                                }
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s.empty[slot]);
            }
            // this warp's partial sums for the block's 32 rows
            float *pb = s.part + (size_t)buf * (NC * M * TCH * 32);
#pragma unroll
            for (int m = 0; m < M; ++m)
#pragma unroll
                for (int t = 0; t < TCH; ++t)
                    if (t < nt)
                        pb[((warp * M + m) * TCH + t) * 32 + lane] = acc[m][t];
            // every consumer reaches this barrier once per chunk, aborted or not; a warp
            // that aborts sets the flag first, so all of them leave together
            named_sync(1, NT);
            if (aborted || *reinterpret_cast<volatile int *>(s.abort_flag))
                return;
            for (int t = warp; t < nt; t += NC) {
                if (MODE == MODE_GATEUP) {
                    float gt = 0.0f, up = 0.0f;
                    for (int w = 0; w < NC; ++w) {
                        gt += pb[((w * 2 + 0) * TCH + t) * 32 + lane];
                        up += pb[((w * 2 + 1) * TCH + t) * 32 + lane];
                    }
                    const float h = gt / (1.0f + expf(-gt)) * up;
                    const float amax = warp_max(fabsf(h));
                    const float dd = __fdiv_rn(amax, 127.0f);
                    const int q = q8_code(h, dd);
                    const long r = s.orow[t];
                    const long hb = r * a.fmax + (long)it.rb * G;
                    a.hq[hb + lane] = (int8_t)q;
                    a.hq_eo[hb + eo_pos(lane)] = (int8_t)q;
                    const int sq = warp_sum_i(q);
                    if (lane == 0) {
                        const int fsg = a.fmax / G;
                        a.hs[r * fsg + it.rb] = dd;
                        a.hc[r * fsg + it.rb] = 8 * sq;
                    }
                } else {
                    float y = 0.0f;
                    for (int w = 0; w < NC; ++w)
                        y += pb[(w * TCH + t) * 32 + lane];
                    a.y[(long)s.orow[t] * a.d + (long)it.rb * G + lane] = y;
                }
            }
            buf ^= 1;
        }
    }
}

// ---- host-side dispatch -----------------------------------------------------------

namespace {

constexpr int RING_NC = 16;             // consumer warps
constexpr size_t RING_BUDGET = 220 * 1024;

// Groups per consumer warp and stage: stages of about 40 KB.
template <int MODE>
constexpr int ring_gpw()
{
    return MODE == MODE_GATEUP ? 2 : 4;
}

template <int MODE, int TCH>
cudaError_t launch_ring(DecodeArgs a, int max_items, cudaStream_t s)
{
    constexpr int M = MODE == MODE_GATEUP ? 2 : 1;
    auto fn = k_ring<MODE, RING_NC, TCH, ring_gpw<MODE>()>;
    a.sg = RING_NC * ring_gpw<MODE>();
    a.stage_bytes = M * a.sg * (512 + 128);
    const size_t fixed = ring_fixed_bytes(a.kmax, RING_NC, M, TCH, 16);
    if (fixed + 2 * (size_t)a.stage_bytes > RING_BUDGET)
        return cudaErrorInvalidValue;
    int ns = (int)((RING_BUDGET - fixed) / a.stage_bytes);
    a.ring = ns > 16 ? 16 : ns;
    const size_t smem = (size_t)a.ring * a.stage_bytes + ring_fixed_bytes(a.kmax, RING_NC, M, TCH, a.ring);
    int dev = 0, n_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int grid = max_items < n_sm ? max_items : n_sm;
    fn<<<grid, (RING_NC + 1) * 32, smem, s>>>(a);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const DecodeArgs &a, int max_items, cudaStream_t s)
{
    switch (a.tch) {
    case 1: return launch_ring<MODE, 1>(a, max_items, s);
    case 2: return launch_ring<MODE, 2>(a, max_items, s);
    case 4: return launch_ring<MODE, 4>(a, max_items, s);
    default: return launch_ring<MODE, 8>(a, max_items, s);
    }
}

}  // namespace

cudaError_t launch_decode(int mode, DecodeArgs a, int max_items, cudaStream_t s)
{
    if (max_items <= 0)
        return cudaSuccess;
    a.kmax = mode == MODE_GATEUP ? a.d : a.fmax;
    const int tmax = a.T < 8 ? a.T : 8;
    a.tch = tmax <= 1 ? 1 : tmax <= 2 ? 2 : tmax <= 4 ? 4 : 8;
    return mode == MODE_GATEUP ? launch_mode<MODE_GATEUP>(a, max_items, s)
                               : launch_mode<MODE_DOWN>(a, max_items, s);
}

}  // namespace clb
