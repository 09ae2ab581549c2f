// Decode GEMVs that stream expert weights through a shared-memory ring.
//
// One persistent CTA per SM walks a list of work items (a block of rows of one expert
// slot). A producer warp copies each item's weight rows and their group scales into a
// ring of NS stages with 1-D bulk copies (cp.async.bulk, completion counted on a "full"
// mbarrier per stage), so that many copies are in flight per SM at any time; consumer
// warps take a stage, compute int32 group dots of the nibbles against the activation
// codes they hold in registers, and release the stage on its "empty" mbarrier.
//
// Lane <-> group mapping: within a K-slice of 32*GPL groups, lane l owns groups
// l, l+32, ...; a lane keeps the even/odd-ordered codes, the scale and the +8 correction
// of its groups for up to TC tokens in registers, and reads 16 bytes of nibbles and one
// scale per group and row from shared memory (512 contiguous bytes per warp: no bank
// conflicts). The per-lane partial sums of a warp are folded by a transpose reduction
// (each shuffle step halves the values a lane carries) instead of one butterfly per value.
//
//   gate/up (MODE_GATEUP): item = 32 rows of W1 and of W3 (one group of h); consumer warp
//     (ks, j) takes row j of both matrices in each stage for K-slice ks; after the last
//     stage the K-slice partials are summed in a fixed order, h = silu(gate) * up is
//     formed and quantised (q8 over the 32 rows, one warp per token).
//   down (MODE_DOWN): item = 64 rows of W2; one K-slice; warp j takes rows j and j+MR of
//     each stage and writes y[pair][row] directly.
#include "kernels.cuh"

namespace clb {

namespace {

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Sum of v[i] over the 32 lanes for N values (N a power of two <= 32). Each of the first
// log2(N) shuffle steps sends half of the values a lane carries to its partner and keeps
// the other half, so a lane ends with one value: the total of value index lane >> (5 -
// log2 N). The remaining steps are a plain butterfly.
template <int N>
__device__ __forceinline__ float xreduce(float (&v)[N], int lane)
{
    int o = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL, send, o);
        }
        o >>= 1;
    }
    float r = v[0];
    for (; o > 0; o >>= 1)
        r += __shfl_xor_sync(FULL, r, o);
    return r;
}

__host__ __device__ constexpr int up16(int n)
{
    return (n + 15) & ~15;
}

template <int N>
__host__ __device__ constexpr int ilog2()
{
    return N <= 1 ? 0 : 1 + ilog2<N / 2>();
}

struct ItemInfo {
    colibri_expert ex;
    int is_shared;
    int row0;     // first weight row of the item
    int nrows;    // valid rows of the item (<= item rows)
    int kdim;     // K of the matrix (d for gate/up, f of the slot for down)
    int begin, count;
};

template <int MODE>
__device__ __forceinline__ ItemInfo item_info(const StreamArgs &a, int item)
{
    ItemInfo it;
    int slot, rb;
    if (MODE == MODE_GATEUP) {
        const int sh_items = a.has_shared ? a.shared_ffn / G : 0;
        if (item < sh_items) {
            slot = 0;
            rb = item;
        } else {
            const int r = item - sh_items, nrb = a.ffn / G;
            slot = (a.has_shared ? 1 : 0) + r / nrb;
            rb = r % nrb;
        }
        it.row0 = rb * G;
        it.nrows = G;
        it.kdim = a.d;
    } else {
        const int nmb = (a.d + DN_ITEM_ROWS - 1) / DN_ITEM_ROWS;
        slot = item / nmb;
        rb = item % nmb;
        it.row0 = rb * DN_ITEM_ROWS;
        it.nrows = min(DN_ITEM_ROWS, a.d - it.row0);
    }
    const Slot sd = a.slots[slot];
    it.is_shared = sd.expert < 0;
    it.ex = it.is_shared ? a.shared : a.experts[sd.expert];
    it.begin = sd.begin;
    it.count = sd.count;
    if (MODE == MODE_DOWN)
        it.kdim = it.is_shared ? a.shared_ffn : a.ffn;
    return it;
}

}  // namespace

// Template parameters: GPL groups per lane, NKS K-slices, MR consumer warps per K-slice,
// TC tokens per register chunk. Block = (NKS*MR + 1) warps; the last warp produces.
template <int MODE, int GPL, int NKS, int MR, int TC>
__global__ void __launch_bounds__((NKS * MR + 1) * 32, 1) k_stream(StreamArgs a)
{
    extern __shared__ __align__(128) unsigned char sm[];
    constexpr int NCW = NKS * MR;                 // consumer warps
    constexpr int SR = MODE == MODE_GATEUP ? MR : 2 * MR;  // rows per matrix per stage
    constexpr int IR = MODE == MODE_GATEUP ? G : DN_ITEM_ROWS;  // rows per item
    constexpr int SPI = IR / SR;                  // stages per item
    constexpr int NV = 2 * TC;                    // values a warp reduces per stage and chunk
    constexpr int LNV = ilog2<NV>();
    const int NS = a.ring;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Counters ct = *a.counters;
    const int n_items = MODE == MODE_GATEUP ? ct.n_items_gateup : ct.n_items_down;

    unsigned char *ring = sm;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)NS * a.stage_bytes);
    uint64_t *empty = full + NS;
    int *abort_flag = reinterpret_cast<int *>(empty + NS);
    float *part = reinterpret_cast<float *>(sm + (size_t)NS * a.stage_bytes + 16 * NS + 16);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ---------------- producer ----------------
        if (lane != 0)
            return;
        uint32_t st = 0;
        // On an abort, wait (bounded) for the copies this thread issued, so that none is
        // still writing into the ring when the CTA exits.
        auto drain = [&]() {
            const uint32_t n = st < (uint32_t)NS ? st : (uint32_t)NS;
            for (uint32_t k = 1; k <= n; ++k) {
                const uint32_t q = st - k;
                mbar_wait(&full[q % NS], (q / NS) & 1);
            }
        };
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            const ItemInfo it = item_info<MODE>(a, item);
            const int kb = it.kdim / 2;          // nibble bytes per row
            const int sb = it.kdim / G * 4;      // scale bytes per row
            const int nch = MODE == MODE_GATEUP ? (it.count + a.tpad - 1) / a.tpad : 1;
            for (int s = 0; s < SPI * nch; ++s, ++st) {
                const int slot = st % NS;
                if (st >= (uint32_t)NS && !mbar_wait(&empty[slot], ((st / NS) - 1) & 1)) {
                    atomicOr(a.err, ERR_WAIT_TIMEOUT);
                    *reinterpret_cast<volatile int *>(abort_flag) = 1;
                    drain();
                    return;
                }
                if (*reinterpret_cast<volatile int *>(abort_flag)) {
                    drain();
                    return;
                }
                const int r0 = it.row0 + (s % SPI) * SR;
                const int rows = max(0, min(SR, it.row0 + it.nrows - r0));
                unsigned char *dst = ring + (size_t)slot * a.stage_bytes;
                if (MODE == MODE_GATEUP) {
                    const uint32_t wb = (uint32_t)(rows * kb), scb = (uint32_t)(rows * sb);
                    mbar_arrive_expect_tx(&full[slot], 2 * wb + 2 * scb);
                    if (rows > 0) {
                        bulk_g2s(dst, it.ex.w1 + (long)r0 * kb, wb, &full[slot]);
                        bulk_g2s(dst + SR * kb, it.ex.w3 + (long)r0 * kb, wb, &full[slot]);
                        bulk_g2s(dst + 2 * SR * kb, it.ex.s1 + (long)r0 * (sb / 4), scb, &full[slot]);
                        bulk_g2s(dst + 2 * SR * kb + up16(SR * sb), it.ex.s3 + (long)r0 * (sb / 4), scb,
                                 &full[slot]);
                    }
                } else {
                    const uint32_t wb = (uint32_t)(rows * kb), scb = (uint32_t)(rows * sb);
                    mbar_arrive_expect_tx(&full[slot], wb + scb);
                    if (rows > 0) {
                        bulk_g2s(dst, it.ex.w2 + (long)r0 * kb, wb, &full[slot]);
                        bulk_g2s(dst + SR * kb, it.ex.s2 + (long)r0 * (sb / 4), scb, &full[slot]);
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int ks = warp / MR, j = warp % MR;
    const int ngs_x = a.act_groups;  // scale/correction stride of the activation rows
    uint32_t st = 0;
    int buf = 0;
    bool aborted = false;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const ItemInfo it = item_info<MODE>(a, item);
        const int kb = it.kdim / 2, sb = it.kdim / G * 4, ng = it.kdim / G;
        // gate/up: the slot's tokens in chunks of tpad (the partial buffers hold tpad); the
        // weights of the item are streamed once per chunk
        const int nch = MODE == MODE_GATEUP ? (it.count + a.tpad - 1) / a.tpad : 1;
        for (int ch = 0; ch < nch; ++ch) {
        const int cb = MODE == MODE_GATEUP ? ch * a.tpad : 0;
        const int npart = MODE == MODE_GATEUP ? min(a.tpad, it.count - cb) : it.count;
        float *pbuf = part + (size_t)buf * (NKS * 2 * a.tpad * G);
        // A chunk of at most TC tokens (the usual decode case) keeps its activation codes in
        // registers for all stages of the item: they are loaded once, before the first wait
        // on the ring, so their latency hides behind it. Larger chunks reload per stage.
        const bool cached = npart <= TC;
        uint4 XA0[TC][GPL], XA1[TC][GPL];
        int XC[TC][GPL];
        float XS[TC][GPL];
#pragma unroll
        for (int t = 0; t < TC; ++t) {
            long arow = 0;
            if (cached && t < npart) {
                const int cs = cb + t;
                if (MODE == MODE_GATEUP)
                    arow = it.is_shared ? cs : a.pairs[it.begin + cs] / a.K;
                else
                    arow = it.is_shared ? (long)a.T * a.K + cs : a.pairs[it.begin + cs];
            }
#pragma unroll
            for (int i = 0; i < GPL; ++i) {
                const int g = ks * 32 * GPL + i * 32 + lane;
                if (cached && t < npart && g < ng) {
                    const int8_t *xa = a.aq_eo + arow * a.act_stride + g * G;
                    XA0[t][i] = ld_nc(xa);
                    XA1[t][i] = ld_nc(xa + 16);
                    XC[t][i] = a.ac[arow * ngs_x + g];
                    XS[t][i] = a.as[arow * ngs_x + g];
                } else {
                    XA0[t][i] = XA1[t][i] = make_uint4(0, 0, 0, 0);
                    XC[t][i] = 0;
                    XS[t][i] = 0.0f;
                }
            }
        }
        for (int s = 0; s < SPI; ++s, ++st) {
            const int slot = st % NS;
            if (!mbar_wait(&full[slot], (st / NS) & 1)) {
                if (lane == 0)
                    atomicOr(a.err, ERR_WAIT_TIMEOUT);
                *reinterpret_cast<volatile int *>(abort_flag) = 1;
                aborted = true;
                break;
            }
            const unsigned char *stg = ring + (size_t)slot * a.stage_bytes;
            const int r0 = s * SR;  // stage's first row within the item
            // weights of this warp's two row-dots (gate/up: W1 and W3 row j; down: rows j, j+MR)
            uint4 wv[2][GPL];
            float sw[2][GPL];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int row = MODE == MODE_GATEUP ? j : j + b * MR;
                const unsigned char *wrow =
                    stg + (MODE == MODE_GATEUP ? (size_t)b * SR * kb : 0) + (size_t)row * kb;
                const float *srow = reinterpret_cast<const float *>(
                    stg + (MODE == MODE_GATEUP ? 2 * SR * kb + (size_t)b * up16(SR * sb) : (size_t)SR * kb) +
                    (size_t)row * sb);
                const bool row_ok = it.row0 + r0 + row < it.row0 + it.nrows;
#pragma unroll
                for (int i = 0; i < GPL; ++i) {
                    const int g = ks * 32 * GPL + i * 32 + lane;
                    if (row_ok && g < ng) {
                        wv[b][i] = *reinterpret_cast<const uint4 *>(wrow + g * 16);
                        sw[b][i] = srow[g];
                    } else {
                        wv[b][i] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
                        sw[b][i] = 0.0f;
                    }
                }
            }
            for (int c0 = 0; c0 < npart; c0 += TC) {
                float v[NV];
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    v[i] = 0.0f;
#pragma unroll
                for (int t = 0; t < TC; ++t) {
                    const int c = c0 + t;
                    if (c < npart) {
                        const int cs = cb + c;  // index within the slot
                        long arow = 0;  // activation row: token (gate/up) or pair (down)
                        if (!cached) {
                            if (MODE == MODE_GATEUP)
                                arow = it.is_shared ? cs : a.pairs[it.begin + cs] / a.K;
                            else
                                arow = it.is_shared ? (long)a.T * a.K + cs : a.pairs[it.begin + cs];
                        }
#pragma unroll
                        for (int i = 0; i < GPL; ++i) {
                            const int g = ks * 32 * GPL + i * 32 + lane;
                            if (g < ng) {
                                uint4 A0 = XA0[t][i], A1 = XA1[t][i];
                                int corr = XC[t][i];
                                float sa = XS[t][i];
                                if (!cached) {
                                    const int8_t *xa = a.aq_eo + arow * a.act_stride + g * G;
                                    A0 = ld_nc(xa);
                                    A1 = ld_nc(xa + 16);
                                    corr = a.ac[arow * ngs_x + g];
                                    sa = a.as[arow * ngs_x + g];
                                }
#pragma unroll
                                for (int b = 0; b < 2; ++b) {
                                    const int D = dot_group(wv[b][i], A0, A1, corr);
                                    v[b * TC + t] = fmaf((float)D, sw[b][i] * sa, v[b * TC + t]);
                                }
                            }
                        }
                    }
                }
                const float r = xreduce<NV>(v, lane);
                const int idx = lane >> (5 - LNV);
                const int b = idx / TC, t = idx % TC, c = c0 + t;
                if ((lane & ((1 << (5 - LNV)) - 1)) == 0 && c < npart) {
                    if (MODE == MODE_GATEUP) {
                        pbuf[((ks * 2 + b) * a.tpad + c) * G + r0 + j] = r;
                    } else {
                        const int row = it.row0 + r0 + j + b * MR;
                        if (row < it.row0 + it.nrows) {
                            const long pr = it.is_shared ? (long)a.T * a.K + cb + c : a.pairs[it.begin + cb + c];
                            a.y[pr * a.d + row] = r;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
        }
        if (MODE == MODE_DOWN && aborted)
            goto done;
        if (MODE == MODE_GATEUP) {
            // Every consumer warp reaches this barrier once per chunk, aborted or not; a warp
            // that aborts sets the flag before arriving, so all of them leave together.
            named_sync(1, NCW * 32);
            if (*reinterpret_cast<volatile int *>(abort_flag))
                goto done;
            // h = silu(gate) * up over the item's 32 rows, q8 per token (lane = row)
            const int fsg = a.fmax / G, rb = it.row0 / G;
            for (int c = warp; c < npart; c += NCW) {
                float gt = 0.0f, up = 0.0f;
#pragma unroll
                for (int k = 0; k < NKS; ++k) {
                    gt += pbuf[((k * 2 + 0) * a.tpad + c) * G + lane];
                    up += pbuf[((k * 2 + 1) * a.tpad + c) * G + lane];
                }
                const float h = gt / (1.0f + expf(-gt)) * up;
                const float amax = warp_max(fabsf(h));
                const float dd = __fdiv_rn(amax, 127.0f);
                const int q = q8_code(h, dd);
                const long r = it.is_shared ? (long)a.T * a.K + cb + c : a.pairs[it.begin + cb + c];
                const long hb = r * a.fmax + it.row0;
                a.hq[hb + lane] = (int8_t)q;
                a.hq_eo[hb + eo_pos(lane)] = (int8_t)q;
                const int sq = warp_sum_i(q);
                if (lane == 0) {
                    a.hs[r * fsg + rb] = dd;
                    a.hc[r * fsg + rb] = 8 * sq;
                }
            }
            buf ^= 1;
        }
        }
    }
done:
    return;
}

// ---- host-side dispatch -----------------------------------------------------------

namespace {

struct StreamShape {
    int gpl, nks, mr;
};

StreamShape gateup_shape(int d)
{
    // K-slices of 32*GPL groups times MR row warps. Nine warps (eight consumers and the
    // producer) leave 168 registers a thread, seven leave 255: the 192-group and 256-group
    // shapes use six or eight consumers with two groups a lane when d % 64 == 0 (MR = 2
    // keeps the scale rows of a stage 16-byte aligned only then).
    const int ng = d / G;
    if (ng <= 32)
        return {1, 1, 8};
    if (ng <= 64)
        return {2, 1, 8};
    if (ng <= 96)
        return {3, 1, 8};
    if (ng <= 128)
        return {2, 2, 4};
    if (ng <= 192)
        return d % 64 == 0 ? StreamShape{2, 3, 2} : StreamShape{3, 2, 4};
    return d % 64 == 0 ? StreamShape{2, 4, 2} : StreamShape{4, 2, 4};
}

int down_gpl(int fmax)
{
    const int ng = fmax / G;
    return ng <= 32 ? 1 : ng <= 64 ? 2 : ng <= 96 ? 3 : 4;
}

// Tokens held in registers per chunk: four, or two when a lane owns three or more groups.
template <int GPL>
constexpr int tc_for()
{
    return GPL <= 2 ? STREAM_TC : 2;
}

template <int MODE, int GPL, int NKS, int MR>
cudaError_t launch_t(const StreamArgs &a, size_t smem, int grid, cudaStream_t s)
{
    auto fn = k_stream<MODE, GPL, NKS, MR, tc_for<GPL>()>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    fn<<<grid, (NKS * MR + 1) * 32, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t stream_stage_bytes(int mode, int d, int fmax)
{
    if (mode == MODE_GATEUP) {
        const StreamShape sh = gateup_shape(d);
        return (size_t)2 * sh.mr * ((size_t)d / 2) + 2 * (size_t)up16(sh.mr * (d / G * 4));
    }
    return (size_t)16 * ((size_t)fmax / 2 + (size_t)fmax / G * 4);
}

// Dynamic shared memory of a launch: ring, barriers (+ abort flag), K-slice partials.
static size_t stream_smem(const StreamArgs &a, int nks)
{
    return (size_t)a.ring * a.stage_bytes + 16 * (size_t)a.ring + 16 +
           (size_t)2 * nks * 2 * a.tpad * G * sizeof(float);
}

cudaError_t launch_stream(int mode, StreamArgs a, int max_items, int n_sm, cudaStream_t s)
{
    constexpr size_t kBudget = 220 * 1024;
    const int nks = mode == MODE_GATEUP ? gateup_shape(a.d).nks : 1;
    a.stage_bytes = (int)stream_stage_bytes(mode, a.d, a.fmax);
    a.tpad = mode == MODE_GATEUP ? (a.T < STREAM_TPAD ? a.T : STREAM_TPAD) : 0;
    a.ring = 2;
    const size_t fixed = stream_smem(a, nks) - 2 * (size_t)a.stage_bytes - 32;
    int ring = (int)((kBudget - fixed) / (a.stage_bytes + 16));
    a.ring = ring > 8 ? 8 : ring;
    if (a.ring < 2)
        return cudaErrorInvalidValue;
    const size_t smem = stream_smem(a, nks);
    const int grid = max_items < n_sm ? max_items : n_sm;
    if (grid <= 0)
        return cudaSuccess;
    if (mode == MODE_GATEUP) {
        const StreamShape sh = gateup_shape(a.d);
        if (sh.nks == 1) {
            if (sh.gpl == 1)
                return launch_t<MODE_GATEUP, 1, 1, 8>(a, smem, grid, s);
            if (sh.gpl == 2)
                return launch_t<MODE_GATEUP, 2, 1, 8>(a, smem, grid, s);
            return launch_t<MODE_GATEUP, 3, 1, 8>(a, smem, grid, s);
        }
        if (sh.mr == 2)
            return sh.nks == 3 ? launch_t<MODE_GATEUP, 2, 3, 2>(a, smem, grid, s)
                               : launch_t<MODE_GATEUP, 2, 4, 2>(a, smem, grid, s);
        if (sh.gpl == 2)
            return launch_t<MODE_GATEUP, 2, 2, 4>(a, smem, grid, s);
        if (sh.gpl == 3)
            return launch_t<MODE_GATEUP, 3, 2, 4>(a, smem, grid, s);
        return launch_t<MODE_GATEUP, 4, 2, 4>(a, smem, grid, s);
    }
    switch (down_gpl(a.fmax)) {
    case 1: return launch_t<MODE_DOWN, 1, 1, 8>(a, smem, grid, s);
    case 2: return launch_t<MODE_DOWN, 2, 1, 8>(a, smem, grid, s);
    case 3: return launch_t<MODE_DOWN, 3, 1, 8>(a, smem, grid, s);
    default: return launch_t<MODE_DOWN, 4, 1, 8>(a, smem, grid, s);
    }
}

}  // namespace clb
