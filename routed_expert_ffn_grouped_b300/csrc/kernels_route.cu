// q8 activation quantiser, router (logits + grouped top-k) and bucketing kernels.
#include "kernels.cuh"

namespace clb {

// ---- q8 ---------------------------------------------------------------------------
// One warp per 32-element group, lane k holds element k. Writes the plain codes and
// scales; optionally also the even/odd-ordered codes and the offset correction
// 8 * sum(codes) the decode GEMV consumes.
__global__ void __launch_bounds__(256) k_q8(Q8Args a)
{
    const int lane = threadIdx.x & 31;
    const long gw = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int ng = a.cols / G;
    if (a.err && blockIdx.x == 0 && threadIdx.x == 0)
        *a.err = 0;  // the first kernel of a layer call clears the flag
    if (gw >= (long)a.rows * ng)
        return;
    const long row = gw / ng;
    const int g = (int)(gw % ng);
    const long base = row * a.cols + (long)g * G;
    const float x = a.x[base + lane];
    const float amax = warp_max(fabsf(x));
    const float d = __fdiv_rn(amax, 127.0f);
    const int q = q8_code(x, d);
    a.q[base + lane] = (int8_t)q;
    if (lane == 0)
        a.scale[row * ng + g] = d;
    if (a.q_eo) {
        a.q_eo[base + eo_pos(lane)] = (int8_t)q;
        const int s = warp_sum_i(q);
        if (lane == 0)
            a.corr[row * ng + g] = 8 * s;
    }
}

// ---- router logits ----------------------------------------------------------------
// One warp per expert row of Wr (staged in shared memory by a bulk copy), all T tokens.
// Lane j runs the fmaf chain over k = j, j+32, ... ascending for each token, then the
// warp joins the 32 chains with a butterfly (offsets 16, 8, 4, 2, 1); lane 0 holds the
// same value as the halving tree (fp32 addition is commutative).
__global__ void __launch_bounds__(32) k_router_logits(RouterArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *wrow = reinterpret_cast<float *>(smem_raw);
    __shared__ __align__(8) uint64_t bar;
    const int e = blockIdx.x;
    const int lane = threadIdx.x;
    const int d = a.d;
    if (lane == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint32_t bytes = (uint32_t)d * 4u;
    if (lane == 0) {
        mbar_arrive_expect_tx(&bar, bytes);
        const char *src = reinterpret_cast<const char *>(a.Wr + (long)e * d);
        for (uint32_t off = 0; off < bytes; off += 32768u) {
            uint32_t n = bytes - off < 32768u ? bytes - off : 32768u;
            bulk_g2s(reinterpret_cast<char *>(wrow) + off, src + off, n, &bar);
        }
    }
    if (!mbar_wait(&bar, 0)) {
        if (lane == 0 && a.err)
            atomicOr(a.err, ERR_WAIT_TIMEOUT);
        mbar_wait(&bar, 0);  // bounded second wait for the copy still in flight
        return;
    }
    constexpr int TT = 8;
    for (int t0 = 0; t0 < a.T; t0 += TT) {
        float acc[TT];
#pragma unroll
        for (int i = 0; i < TT; ++i)
            acc[i] = 0.0f;
        const int nt = min(TT, a.T - t0);
        for (int k = lane; k < d; k += 32) {
            const float wv = wrow[k];
#pragma unroll
            for (int i = 0; i < TT; ++i)
                if (i < nt)
                    acc[i] = fmaf(__ldg(a.x + (long)(t0 + i) * d + k), wv, acc[i]);
        }
#pragma unroll
        for (int i = 0; i < TT; ++i) {
            float v = acc[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                v = v + __shfl_xor_sync(FULL, v, o);
            if (lane == 0 && i < nt)
                a.logits[(long)(t0 + i) * a.E + e] = v;
        }
    }
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

// ---- router selection -------------------------------------------------------------
// One warp per token. Lane j owns experts e = j + 32 r. Group scores are computed by
// one lane per group over the group's contiguous experts (staged in shared memory);
// group and expert top-k are warp-shuffle argmax rounds with the (value, index) order.
constexpr int SEL_WARPS = 4;

__global__ void __launch_bounds__(32 * SEL_WARPS) k_router_select(SelectArgs a)
{
    __shared__ float s_c[SEL_WARPS][1024];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * SEL_WARPS + w;
    if (t >= a.T)
        return;
    const int E = a.E, R = (E + 31) / 32;
    const float *l = a.logits + (long)t * E;
    float sv[32], cv[32];
    bool avail[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        sv[r] = 0.0f;
        cv[r] = 0.0f;
        avail[r] = false;
        const int e = lane + 32 * r;
        if (r < R && e < E) {
            const float lv = l[e];
            if (a.router == COLIBRI_ROUTER_SOFTMAX) {
                sv[r] = lv;
                cv[r] = lv;
            } else {
                sv[r] = (float)(1.0 / (1.0 + exp(-(double)lv)));
                cv[r] = sv[r] + (a.bias ? a.bias[e] : 0.0f);
            }
            avail[r] = true;
            s_c[w][e] = cv[r];
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
                const float v = s_c[w][lane * gs + i];
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
    // top-k: k rounds of warp argmax over the remaining candidates
    const int K = a.K;
    double sel_sum = 0.0;
    int picks[32];
    float pick_s[32];
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
        const int src = wi >= 0 ? (wi & 31) : 0;
        s_pick = __shfl_sync(FULL, s_pick, src);
        picks[i < 32 ? i : 31] = wi;
        pick_s[i < 32 ? i : 31] = s_pick;
    }
    if (a.router == COLIBRI_ROUTER_SOFTMAX) {
        // softmax over all E logits in fp64
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
        double sel = 0.0;
        for (int i = 0; i < K; ++i)
            sel += exp((double)pick_s[i] - m) / z;
        if (lane == 0) {
            for (int i = 0; i < K; ++i) {
                double p = exp((double)pick_s[i] - m) / z;
                if (a.norm_topk)
                    p = p / sel;
                a.ids[(long)t * K + i] = picks[i];
                a.w[(long)t * K + i] = (float)(p * (double)a.routed_scale);
            }
        }
    } else {
        for (int i = 0; i < K; ++i)
            sel_sum += (double)pick_s[i];
        if (lane == 0) {
            for (int i = 0; i < K; ++i) {
                double p = (double)pick_s[i];
                if (a.norm_topk)
                    p = p / sel_sum;
                a.ids[(long)t * K + i] = picks[i];
                a.w[(long)t * K + i] = (float)(p * (double)a.routed_scale);
            }
        }
    }
}

// ---- bucketing --------------------------------------------------------------------
// One CTA of 1024 threads. Counts per expert (shared-memory atomics), exclusive scan,
// then a stable scatter in chunks of 1024 pairs: a pair's position is its expert's
// running base + the count of the same expert in earlier warps of the chunk + its rank
// among equal lanes of its warp (__match_any_sync). Finally the slot list (shared
// expert first, then routed experts in ascending id) and the item counts.
__global__ void __launch_bounds__(1024) k_bucket(BucketArgs a)
{
    extern __shared__ int sm[];
    const int E = a.E;
    int *cnt = sm;              // [E]
    int *run = sm + E;          // [E]
    int *wcnt = sm + 2 * E;     // [32][E]
    __shared__ int s_warp[32];
    __shared__ int s_total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long P = (long)a.T * a.K;
    for (int e = tid; e < E; e += 1024)
        cnt[e] = 0;
    __syncthreads();
    for (long p = tid; p < P; p += 1024) {
        const int e = a.ids[p];
        if (e < 0 || e >= E) {
            if (a.err)
                atomicOr(a.err, ERR_BAD_ID);
        }
        else
            atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive scan of cnt over E <= 1024 (one element per thread)
    const int c = tid < E ? cnt[tid] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = s_warp[lane];
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(FULL, inc, o);
            if (lane >= o)
                inc += u;
        }
        s_warp[lane] = inc - v;
        if (lane == 31)
            s_total = inc;
    }
    __syncthreads();
    const int excl = incl - c + s_warp[warp];
    if (tid < E) {
        a.offsets[tid] = excl;
        run[tid] = excl;
    }
    if (tid == 0)
        a.offsets[E] = s_total;
    __syncthreads();
    // stable scatter
    for (long base = 0; base < P; base += 1024) {
        for (int i = tid; i < 32 * E; i += 1024)
            wcnt[i] = 0;
        __syncthreads();
        const long p = base + tid;
        int e = p < P ? a.ids[p] : -1;
        if (e < 0 || e >= E)
            e = -1;
        const unsigned m = __match_any_sync(FULL, e);
        const int leader = __ffs(m) - 1;
        const int rank = __popc(m & ((1u << lane) - 1u));
        if (e >= 0 && lane == leader)
            wcnt[warp * E + e] = __popc(m);
        __syncthreads();
        int tot = 0;
        if (tid < E) {
            for (int ww = 0; ww < 32; ++ww) {
                const int v = wcnt[ww * E + tid];
                wcnt[ww * E + tid] = tot;
                tot += v;
            }
        }
        __syncthreads();
        if (e >= 0)
            a.pairs[run[e] + wcnt[warp * E + e] + rank] = (int)p;
        __syncthreads();
        if (tid < E)
            run[tid] += tot;
        __syncthreads();
    }
    // slots: flags scan over experts with a non-zero count
    const int flag = (tid < E && c > 0) ? 1 : 0;
    int fin = flag;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, fin, o);
        if (lane >= o)
            fin += v;
    }
    __syncthreads();
    if (lane == 31)
        s_warp[warp] = fin;
    __syncthreads();
    if (warp == 0) {
        int v = s_warp[lane];
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(FULL, inc, o);
            if (lane >= o)
                inc += u;
        }
        s_warp[lane] = inc - v;
        if (lane == 31)
            s_total = inc;
    }
    __syncthreads();
    const int sbase = a.has_shared ? 1 : 0;
    if (flag) {
        Slot s;
        s.expert = tid;
        s.begin = excl;
        s.count = c;
        s.pad = 0;
        a.slots[sbase + fin - flag + s_warp[warp]] = s;
    }
    if (tid == 0) {
        const int n_routed = s_total;
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
        *a.counters = ct;
    }
}

}  // namespace clb
