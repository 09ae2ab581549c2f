// q8 activation quantiser, router (logits + grouped top-k) and bucketing kernels.
#include "kernels.cuh"

namespace clb {

// ---- q8 ---------------------------------------------------------------------------
// One warp per group of a.group (32 or 64) elements, lane k holding element k (and
// k + 32). Writes the plain codes and scales; optionally also the even/odd-ordered codes
// and the offset correction 8 * sum(codes) per 32 elements that the decode GEMV consumes,
// and the bf16 codes.
__device__ __forceinline__ void q8_group(const Q8Args &a, long gw, int lane);

__global__ void __launch_bounds__(256) k_q8(Q8Args a)
{
    grid_dep_launch();  // a decode expert kernel after this one may be scheduled now
    const int lane = threadIdx.x & 31;
    const long gw = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= a.rows * (a.cols / a.group))
        return;
    q8_group(a, gw, lane);
}

// ---- router logits (+ the fp64 sigmoid, + q8 of x as a side job) --------------------
// One CTA per expert e. The CTA bulk-copies Wr[e] and a chunk of xt token rows of x
// (contiguous in x) into shared memory, then warp w takes the chunk's tokens w, w+nw,
// ...: lane j runs the fmaf chain over k = j, j+32, ... ascending, and the warp joins the
// 32 chains with a butterfly (offsets 16, 8, 4, 2, 1); lane 0 then holds the value of the
// halving tree (fp32 addition is commutative). In sigmoid mode lane 0 also evaluates
// s = fp32(1/(1+exp(-l))) in fp64 and c = s + bias[e], so that the fp64 work is spread
// over all CTAs. Before that, the CTAs quantise x (one warp per 32-group) when the layer
// asks for it.
__device__ __forceinline__ void q8_group(const Q8Args &a, long gw, int lane)
{
    const int gq = a.group, ng = a.cols / gq, halves = gq / G;
    const long row = gw / ng;
    const int g = (int)(gw % ng);
    const long base = row * a.cols + (long)g * gq;
    float x[2];
    float m = 0.0f;
    for (int h = 0; h < halves; ++h) {
        x[h] = a.x[base + h * G + lane];
        m = fmaxf(m, fabsf(x[h]));
    }
    const float amax = warp_max(m);
    const float d = __fdiv_rn(amax, 127.0f), rd = __frcp_rn(d);
    if (lane == 0)
        a.scale[row * ng + g] = d;
    for (int h = 0; h < halves; ++h) {
        const long b = base + h * G;
        const int q = q8_code_r(x[h], d, rd);
        a.q[b + lane] = (int8_t)q;
        if (a.q_bf)
            a.q_bf[b + bf16_pos(lane)] = bf16_of_int(q);
        if (a.q_eo) {
            a.q_eo[b + eo_pos(lane)] = (int8_t)q;
            const int s = warp_sum_i(q);
            if (lane == 0)
                a.corr[row * (a.cols / G) + (long)g * halves + h] = 8 * s;
        }
    }
}

// Returns false if a bulk copy did not land within the wait limit (flagged in a.err).
__device__ bool route_logits_part(const RouterArgs &a, unsigned char *smem_raw, uint64_t *bar)
{
    const int d = a.d, e = blockIdx.x, nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *wrow = reinterpret_cast<float *>(smem_raw);
    float *xs = wrow + d;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // q8 side job: warp-granular, grid-strided over the T*d/32 groups of x
    if (a.q8.x) {
        const long n = (long)a.T * (d / a.q8.group);
        for (long gw = (long)blockIdx.x * nw + warp; gw < n; gw += (long)gridDim.x * nw)
            q8_group(a.q8, gw, lane);
    }
    const uint32_t row_bytes = (uint32_t)d * 4u;
    uint32_t phase = 0;
    for (int t0 = 0; t0 < a.T; t0 += a.xt) {
        const int nt = min(a.xt, a.T - t0);
        if (threadIdx.x == 0) {
            const uint32_t xbytes = row_bytes * (uint32_t)nt;
            mbar_arrive_expect_tx(bar, (t0 == 0 ? row_bytes : 0u) + xbytes);
            if (t0 == 0) {
                const char *src = reinterpret_cast<const char *>(a.Wr + (long)e * d);
                for (uint32_t off = 0; off < row_bytes; off += 32768u)
                    bulk_g2s(reinterpret_cast<char *>(wrow) + off, src + off, min(32768u, row_bytes - off), bar);
            }
            const char *xsrc = reinterpret_cast<const char *>(a.x + (long)t0 * d);
            for (uint32_t off = 0; off < xbytes; off += 32768u)
                bulk_g2s(reinterpret_cast<char *>(xs) + off, xsrc + off, min(32768u, xbytes - off), bar);
        }
        if (!mbar_wait(bar, phase)) {
            if (lane == 0 && a.err)
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
            mbar_wait(bar, phase);  // bounded second wait for the copies still in flight
            return false;
        }
        phase ^= 1u;
        for (int i = warp; i < nt; i += nw) {
            const float *xr = xs + (long)i * d;
            float acc = 0.0f;
#pragma unroll 8
            for (int k = lane; k < d; k += 32)
                acc = fmaf(xr[k], wrow[k], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc = acc + __shfl_xor_sync(FULL, acc, o);
            if (lane == 0) {
                const long o = (long)(t0 + i) * a.E + e;
                a.logits[o] = acc;
                if (a.s) {
                    const float sv = (float)(1.0 / (1.0 + exp(-(double)acc)));
                    a.s[o] = sv;
                    a.c[o] = sv + (a.bias ? a.bias[e] : 0.0f);
                }
            }
        }
        __syncthreads();  // the chunk buffer is refilled next
    }
    return true;
}

// ---- router logits for many tokens: (16 tokens x 32 experts) tiles --------------------
// The same fixed summation order as route_logits_part: lane j of a warp keeps chain j
// (k = j, j+32, ... ascending, fmaf) for each of its (token, expert) pairs; K-chunks of x
// and of Wr are staged in shared memory for the whole CTA by cp.async, two stages deep, so
// that the next chunk's copies run while the current one is summed. Warp w owns experts 4w..4w+3
// of the tile and all 16 tokens: 64 chains a lane. The chains of each pair are then
// added in the halving-tree pairs (16, 8, 4, 2, 1) by a transpose reduction: each step
// adds the same two partial sums as the tree, only in another lane, so the result is the
// tree's bit for bit; lane l ends with pair l and pair 32 + l, and evaluates their
// sigmoid scores (fp64) in parallel.
constexpr int RT_T = 16, RT_E = 32, RT_KC = 256;
static_assert(ROUTE_TILED_SMEM == 2 * (RT_T + RT_E) * RT_KC * sizeof(float), "launch size of the tiled router");

template <int N>
__device__ __forceinline__ float tree_reduce_lanes(float (&v)[N], int lane)
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
    return v[0];
}

__global__ void __launch_bounds__(256, 2) k_route_logits_tiled(RouterArgs a)
{
    extern __shared__ __align__(16) float rt_smem[];  // [2] x (xs [RT_T][RT_KC], ws [RT_E][RT_KC])
    constexpr int STAGE = (RT_T + RT_E) * RT_KC;
    const int d = a.d, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * RT_T, e0 = blockIdx.y * RT_E;
    const int nt = min(RT_T, a.T - t0), ne = min(RT_E, a.E - e0);
    const int nck = (d + RT_KC - 1) / RT_KC;
    // K-chunk c of the tile's rows of x and Wr into stage c & 1; rows past the tile are
    // zero-filled (a copy of 0 source bytes from the tile's first row)
    auto stage_chunk = [&](int c) {
        float *xs = rt_smem + (c & 1) * STAGE, *ws = xs + RT_T * RT_KC;
        const int k0 = c * RT_KC, q = min(RT_KC, d - k0) / 4;
        for (int i = threadIdx.x; i < (RT_T + RT_E) * q; i += blockDim.x) {
            const int r = i / q, col = (i - r * q) * 4;
            if (r < RT_T) {
                const bool live = r < nt;
                cp_async16(xs + r * RT_KC + col, a.x + (long)(t0 + (live ? r : 0)) * d + k0 + col, live ? 16u : 0u);
            } else {
                const int e = r - RT_T;
                const bool live = e < ne;
                cp_async16(ws + e * RT_KC + col, a.Wr + (long)(e0 + (live ? e : 0)) * d + k0 + col, live ? 16u : 0u);
            }
        }
        cp_async_commit();
    };
    float acc[RT_T * 4];  // [expert 4w+i][token t]: index i * 16 + t
#pragma unroll
    for (int i = 0; i < RT_T * 4; ++i)
        acc[i] = 0.0f;
    stage_chunk(0);
    for (int c = 0; c < nck; ++c) {
        if (c + 1 < nck) {
            stage_chunk(c + 1);  // into the stage chunk c - 1 used (freed by the barrier below)
            cp_async_wait_group<1>();
        } else {
            cp_async_wait_group<0>();
        }
        __syncthreads();
        const float(*xs)[RT_KC] = reinterpret_cast<const float(*)[RT_KC]>(rt_smem + (c & 1) * STAGE);
        const float(*ws)[RT_KC] = reinterpret_cast<const float(*)[RT_KC]>(rt_smem + (c & 1) * STAGE + RT_T * RT_KC);
        const int kc = min(RT_KC, d - c * RT_KC);  // a multiple of 32
        for (int k = lane; k < kc; k += 32) {
            float xv[RT_T];
#pragma unroll
            for (int t = 0; t < RT_T; ++t)
                xv[t] = xs[t][k];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float wv = ws[warp * 4 + i][k];
#pragma unroll
                for (int t = 0; t < RT_T; ++t)
                    acc[i * RT_T + t] = fmaf(xv[t], wv, acc[i * RT_T + t]);
            }
        }
        __syncthreads();  // every warp is done with stage c & 1 before chunk c + 2 refills it
    }
    float lo[32], hi[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        lo[i] = acc[i];
        hi[i] = acc[32 + i];
    }
    const float r0 = tree_reduce_lanes<32>(lo, lane);  // pair index lane
    const float r1 = tree_reduce_lanes<32>(hi, lane);  // pair index 32 + lane
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int idx = h * 32 + lane;
        const int t = idx % RT_T, e = warp * 4 + idx / RT_T;
        if (t < nt && e < ne) {
            const float l = h ? r1 : r0;
            const long o = (long)(t0 + t) * a.E + e0 + e;
            a.logits[o] = l;
            if (a.s) {
                const float sv = (float)(1.0 / (1.0 + exp(-(double)l)));
                a.s[o] = sv;
                a.c[o] = sv + (a.bias ? a.bias[e0 + e] : 0.0f);
            }
        }
    }
}

__global__ void __launch_bounds__(128) k_route_logits(RouterArgs a)
{
    grid_dep_launch();  // a decode expert kernel after this one may be scheduled now
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    route_logits_part(a, smem_raw, &bar);
}

// (value, index) order of the selection: larger value first, then lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return bi < 0 || v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float &v, int &i)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(FULL, v, o);
        int oi = __shfl_xor_sync(FULL, i, o);
        if (oi >= 0 && better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

// ---- router selection (one warp per token) ----------------------------------------
// Lane j owns experts e = j + 32 r. Sigmoid mode reads s and c from the logits kernel
// when it wrote them, else evaluates them here the same way;
// group scores are computed by one lane per group over the group's contiguous experts
// (staged in shared memory); group and expert top-k are warp-shuffle argmax rounds with
// the (value, index) order. sc: this warp's shared row of at least E floats.
__device__ void select_token(const SelectArgs &a, int t, int lane, float *sc)
{
    const int E = a.E, R = (E + 31) / 32;
    const long row = (long)t * E;
    float sv[32], cv[32];
    bool avail[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        sv[r] = 0.0f;
        cv[r] = 0.0f;
        avail[r] = false;
        const int e = lane + 32 * r;
        if (r < R && e < E) {
            if (a.router == COLIBRI_ROUTER_SOFTMAX) {
                sv[r] = a.logits[row + e];
                cv[r] = rank_score(sv[r]);
            } else if (a.s) {
                sv[r] = a.s[row + e];
                cv[r] = rank_score(a.c[row + e]);
            } else {
                sv[r] = (float)(1.0 / (1.0 + exp(-(double)a.logits[row + e])));
                cv[r] = rank_score(sv[r] + (a.bias ? a.bias[e] : 0.0f));
            }
            avail[r] = true;
            sc[e] = cv[r];
        }
    }
    __syncwarp();
    if (a.router != COLIBRI_ROUTER_SOFTMAX) {
        // group scores: lane g scans group g for its two largest c
        const int gs = E / a.n_group;
        float gscore = 0.0f;
        int gidx = -1;
        if (lane < a.n_group) {
            float m1 = -INFINITY, m2 = -INFINITY;
            for (int i = 0; i < gs; ++i) {
                const float v = sc[lane * gs + i];
                if (v > m1) {
                    m2 = m1;
                    m1 = v;
                } else if (v > m2) {
                    m2 = v;
                }
            }
            gscore = gs == 1 ? m1 : m1 + m2;
            gidx = lane;
        }
        bool kept = false;
        for (int r = 0; r < a.topk_group; ++r) {
            float bv = gidx >= 0 && !kept ? gscore : 0.0f;
            int bi = gidx >= 0 && !kept ? gidx : -1;
            warp_argmax(bv, bi);
            if (bi == lane)
                kept = true;
        }
        const unsigned keep_mask = __ballot_sync(FULL, kept);
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int e = lane + 32 * r;
            if (avail[r] && !((keep_mask >> (e / gs)) & 1u))
                avail[r] = false;
        }
    }
    // top-k: k rounds of warp argmax over the remaining candidates; lane i keeps pick i
    const int K = a.K;
    int my_pick = -1;
    float my_s = 0.0f;
    for (int i = 0; i < K; ++i) {
        float bv = 0.0f;
        int bi = -1, br = -1;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int e = lane + 32 * r;
            if (avail[r] && better(cv[r], e, bv, bi)) {
                bv = cv[r];
                bi = e;
                br = r;
            }
        }
        float wv = bv;
        int wi = bi;
        warp_argmax(wv, wi);
        float s_pick = 0.0f;
        if (wi == bi && bi >= 0) {
#pragma unroll
            for (int r = 0; r < 32; ++r)
                if (r == br) {
                    avail[r] = false;
                    s_pick = sv[r];
                }
        }
        s_pick = __shfl_sync(FULL, s_pick, wi >= 0 ? (wi & 31) : 0);
        if (lane == i) {
            my_pick = wi;
            my_s = s_pick;
        }
    }
    // weights: lane i < K holds pick i; sums in selection order (lane 0 first)
    double p = (double)my_s, scale_sum = 0.0;
    if (a.router == COLIBRI_ROUTER_SOFTMAX) {
        const float *l = a.logits + row;
        double m = -INFINITY;
        for (int e = lane; e < E; e += 32)
            m = fmax(m, (double)l[e]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = fmax(m, __shfl_xor_sync(FULL, m, o));
        double z = 0.0;
        for (int e = lane; e < E; e += 32)
            z += exp((double)l[e] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            z += __shfl_xor_sync(FULL, z, o);
        p = lane < K ? exp(p - m) / z : 0.0;
    }
    for (int i = 0; i < K; ++i)
        scale_sum += __shfl_sync(FULL, lane < K ? p : 0.0, i);
    if (lane < K) {
        if (a.norm_topk)
            p = p / scale_sum;
        a.ids[(long)t * K + lane] = my_pick;
        a.w[(long)t * K + lane] = (float)(p * (double)a.routed_scale);
    }
}

constexpr int SEL_WARPS = 4;

__global__ void __launch_bounds__(32 * SEL_WARPS) k_router_select(SelectArgs a)
{
    grid_dep_launch();  // a decode expert kernel after this one may be scheduled now
    __shared__ float s_c[SEL_WARPS][1024];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * SEL_WARPS + w;
    if (t >= a.T)
        return;
    select_token(a, t, lane, s_c[w]);
}

// ---- bucketing --------------------------------------------------------------------
// One CTA of 1024 threads. Counts per expert (shared-memory atomics), exclusive scan,
// then a stable scatter in chunks of 1024 pairs: a pair's position is its expert's
// running base + the count of the same expert in earlier warps of the chunk + its rank
// among equal lanes of its warp (__match_any_sync). Finally the slot list (shared
// expert first, then routed experts in ascending id) and the item counts.
// ---- block-wide helpers (any blockDim.x that is a multiple of 32, up to 1024) -------

// In-place exclusive scan of the shared array v[0..n) by the whole block; returns the
// total to every thread. Each thread scans a contiguous run of ceil(n / blockDim.x).
__device__ int block_excl_scan(int *v, int n)
{
    __shared__ int s_w[32];
    __shared__ int s_tot;
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + nt - 1) / nt;
    const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
    int sum = 0;
    for (int i = b0; i < b1; ++i)
        sum += v[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(FULL, incl, o);
        if (lane >= o)
            incl += u;
    }
    if (lane == 31)
        s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nwarps = nt >> 5;
        const int x = lane < nwarps ? s_w[lane] : 0;
        int inc = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(FULL, inc, o);
            if (lane >= o)
                inc += u;
        }
        if (lane < nwarps)
            s_w[lane] = inc - x;
        if (lane == 31)
            s_tot = inc;
    }
    __syncthreads();
    int run = incl - sum + s_w[warp];
    for (int i = b0; i < b1; ++i) {
        const int x = v[i];
        v[i] = run;
        run += x;
    }
    const int tot = s_tot;
    __syncthreads();
    return tot;
}

// ---- bucketing --------------------------------------------------------------------
// Counts per expert (shared-memory atomics), exclusive scan into offsets, then a stable
// scatter in chunks of blockDim.x pairs: a pair's position is its expert's running base
// + the count of the same expert in earlier warps of the chunk + its rank among equal
// lanes of its warp (__match_any_sync). Finally the slot list (shared expert first, then
// the routed experts in ascending id) and the work-item counts. sid: the T*K ids (shared
// or global memory); sm: 3*E + nwarps*E ints of shared memory.
__device__ void bucket_block(const BucketArgs &a, const int32_t *sid, int *sm)
{
    const int E = a.E, nt = blockDim.x, nwarps = nt >> 5;
    int *cnt = sm;               // [E] counts, then offsets
    int *run = sm + E;           // [E]
    int *flag = sm + 2 * E;      // [E] nonzero-count flags, then their exclusive scan
    int *wcnt = sm + 3 * E;      // [nwarps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long P = (long)a.T * a.K;
    for (int e = tid; e < E; e += nt)
        cnt[e] = 0;
    __syncthreads();
    for (long p = tid; p < P; p += nt) {
        const int e = sid[p];
        if (e < 0 || e >= E) {
            if (a.err)
                atomicOr(a.err, ERR_BAD_ID);
        } else {
            atomicAdd(&cnt[e], 1);
            // a token must not list an expert twice
            for (long q = p - p % a.K; q < p; ++q)
                if (sid[q] == e && a.err)
                    atomicOr(a.err, ERR_BAD_ID);
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) {
        flag[e] = cnt[e] > 0;
        run[e] = cnt[e];
    }
    __syncthreads();
    const int total = block_excl_scan(run, E);  // run = offsets
    for (int e = tid; e < E; e += nt) {
        a.offsets[e] = run[e];
        cnt[e] = run[e];  // keep the offsets for the slot list
    }
    if (tid == 0)
        a.offsets[E] = total;
    __syncthreads();
    // stable scatter
    for (long base = 0; base < P; base += nt) {
        for (int i = tid; i < nwarps * E; i += nt)
            wcnt[i] = 0;
        __syncthreads();
        const long p = base + tid;
        int e = p < P ? sid[p] : -1;
        if (e < 0 || e >= E)
            e = -1;
        const unsigned m = __match_any_sync(FULL, e);
        const int leader = __ffs(m) - 1;
        const int rank = __popc(m & ((1u << lane) - 1u));
        if (e >= 0 && lane == leader)
            wcnt[warp * E + e] = __popc(m);
        __syncthreads();
        for (int x = tid; x < E; x += nt) {
            int tot = 0;
            for (int ww = 0; ww < nwarps; ++ww) {
                const int v = wcnt[ww * E + x];
                wcnt[ww * E + x] = tot;
                tot += v;
            }
            flag[x] |= tot << 1;  // chunk total, consumed below
        }
        __syncthreads();
        if (e >= 0)
            a.pairs[run[e] + wcnt[warp * E + e] + rank] = (int)p;
        __syncthreads();
        for (int x = tid; x < E; x += nt) {
            run[x] += flag[x] >> 1;
            flag[x] &= 1;
        }
        __syncthreads();
    }
    // slots: routed experts with a non-zero count, in ascending id after the shared one
    const int n_routed = block_excl_scan(flag, E);
    const int sbase = a.has_shared ? 1 : 0;
    for (int e = tid; e < E; e += nt) {
        const int c = (e + 1 < E ? cnt[e + 1] : total) - cnt[e];
        if (c > 0) {
            Slot s;
            s.expert = e;
            s.begin = cnt[e];
            s.count = c;
            s.pad = 0;
            a.slots[sbase + flag[e]] = s;
        }
    }
    if (tid == 0) {
        if (a.has_shared) {
            Slot s;
            s.expert = -1;
            s.begin = 0;
            s.count = a.T;
            s.pad = 0;
            a.slots[0] = s;
        }
        Counters ct;
        ct.n_slots = sbase + n_routed;
        ct.n_routed = n_routed;
        ct.n_items_gateup = (a.has_shared ? a.shared_ffn / G : 0) + n_routed * (a.ffn / G);
        ct.n_items_down = ct.n_slots * a.down_blocks;
        ct.n_rows = total + (a.has_shared ? a.T : 0);
        ct.pad[0] = ct.pad[1] = ct.pad[2] = 0;
        *a.counters = ct;
    }
}

size_t bucket_smem_bytes(int E, int nthreads)
{
    return (size_t)(3 + nthreads / 32) * E * sizeof(int);
}

// Prefill bucketing: one CTA of 1024 threads; the ids are staged in shared memory after
// the counters when they fit (stage_ids).
__global__ void __launch_bounds__(1024) k_bucket(BucketArgs a)
{
    extern __shared__ int sm[];
    const int32_t *sid = a.ids;
    if (a.stage_ids) {
        int *st = sm + (3 + 32) * a.E;
        const long P = (long)a.T * a.K;
        for (long p = threadIdx.x; p < P; p += blockDim.x)
            st[p] = a.ids[p];
        sid = st;
        __syncthreads();
    }
    bucket_block(a, sid, sm);
}

}  // namespace clb
