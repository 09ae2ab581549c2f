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

// ---- router logits (+ the fp64 sigmoid, + q8 of x as a side job) --------------------
// One CTA per expert e, four warps. The CTA bulk-copies Wr[e] and a chunk of XT token
// rows of x (contiguous in x) into shared memory, then warp w takes the chunk's tokens
// w, w+4, ...: lane j runs the fmaf chain over k = j, j+32, ... ascending, and the warp
// joins the 32 chains with a butterfly (offsets 16, 8, 4, 2, 1); lane 0 then holds the
// value of the halving tree (fp32 addition is commutative). In sigmoid mode lane 0 also
// evaluates s = fp32(1/(1+exp(-l))) in fp64 and c = s + bias[e], so that the fp64 work
// is spread over all CTAs. Before that, the CTAs quantise x (one warp per 32-group) when
// the layer asks for it.
constexpr int RL_WARPS = 4;

__device__ __forceinline__ void q8_group(const Q8Args &a, long gw, int lane)
{
    const int ng = a.cols / G;
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

__global__ void __launch_bounds__(32 * RL_WARPS) k_route_logits(RouterArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    const int d = a.d, e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *wrow = reinterpret_cast<float *>(smem_raw);
    float *xs = wrow + d;
    if (a.err && blockIdx.x == 0 && threadIdx.x == 0)
        *a.err = 0;  // the first kernel of a layer call clears the flag
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // q8 side job: warp-granular, grid-strided over the T*d/32 groups of x
    if (a.q8.x) {
        const long n = (long)a.T * (d / G);
        for (long gw = (long)blockIdx.x * RL_WARPS + warp; gw < n; gw += (long)gridDim.x * RL_WARPS)
            q8_group(a.q8, gw, lane);
    }
    const uint32_t row_bytes = (uint32_t)d * 4u;
    uint32_t phase = 0;
    bool ok = true;
    for (int t0 = 0; t0 < a.T; t0 += a.xt) {
        const int nt = min(a.xt, a.T - t0);
        if (threadIdx.x == 0) {
            const uint32_t xbytes = row_bytes * (uint32_t)nt;
            mbar_arrive_expect_tx(&bar, (t0 == 0 ? row_bytes : 0u) + xbytes);
            if (t0 == 0) {
                const char *src = reinterpret_cast<const char *>(a.Wr + (long)e * d);
                for (uint32_t off = 0; off < row_bytes; off += 32768u)
                    bulk_g2s(reinterpret_cast<char *>(wrow) + off, src + off, min(32768u, row_bytes - off), &bar);
            }
            const char *xsrc = reinterpret_cast<const char *>(a.x + (long)t0 * d);
            for (uint32_t off = 0; off < xbytes; off += 32768u)
                bulk_g2s(reinterpret_cast<char *>(xs) + off, xsrc + off, min(32768u, xbytes - off), &bar);
        }
        if (!mbar_wait(&bar, phase)) {
            ok = false;
            if (lane == 0 && a.err)
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
            mbar_wait(&bar, phase);  // bounded second wait for the copies still in flight
            break;
        }
        phase ^= 1u;
        for (int i = warp; i < nt; i += RL_WARPS) {
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
    (void)ok;
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
                sv[r] = cv[r] = a.logits[row + e];
            } else if (a.s) {
                sv[r] = a.s[row + e];
                cv[r] = a.c[row + e];
            } else {
                sv[r] = (float)(1.0 / (1.0 + exp(-(double)a.logits[row + e])));
                cv[r] = sv[r] + (a.bias ? a.bias[e] : 0.0f);
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
__device__ void bucket_body(const BucketArgs &a, int *sm)
{
    const int E = a.E;
    int *cnt = sm;              // [E]
    int *run = sm + E;          // [E]
    int *wcnt = sm + 2 * E;     // [32][E]
    __shared__ int s_warp[32];
    __shared__ int s_total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long P = (long)a.T * a.K;
    // the ids, staged in shared memory when they fit (the launch sized it so)
    const int32_t *sid = a.ids;
    if (a.stage_ids) {
        int *st = sm + 34 * E;
        for (long p = tid; p < P; p += 1024)
            st[p] = a.ids[p];
        sid = st;
    }
    for (int e = tid; e < E; e += 1024)
        cnt[e] = 0;
    __syncthreads();
    for (long p = tid; p < P; p += 1024) {
        const int e = sid[p];
        if (e < 0 || e >= E) {
            if (a.err)
                atomicOr(a.err, ERR_BAD_ID);
        } else {
            atomicAdd(&cnt[e], 1);
            // a token must not list an expert twice
            const long t0 = p - p % a.K;
            for (long q = t0; q < p; ++q)
                if (sid[q] == e && a.err)
                    atomicOr(a.err, ERR_BAD_ID);
        }
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
        int e = p < P ? sid[p] : -1;
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

__global__ void __launch_bounds__(1024) k_bucket(BucketArgs a)
{
    extern __shared__ int sm[];
    bucket_body(a, sm);
}

// ---- decode selection with the whole CTA -----------------------------------------
// The k-th pick of the sequential selection (repeatedly take the best remaining
// candidate in the (value desc, index asc) order) is the candidate that exactly k others
// beat. So each candidate's thread counts the allowed candidates that beat it and, if
// that rank is below top_k, writes itself to position rank. Groups are kept the same way
// (rank of the group score below topk_group). The CTA (1024 threads) takes TPR tokens per
// round, Epad = E rounded up to 32 threads per token.
//   smem (floats): per token slot c[Epad] | gscore[32] | kept[32] (int) | pick_id[32] (int)
//   | pick_s[32].
constexpr int SEL_SLOT_EXTRA = 128;

__device__ void select_cta(const SelectArgs &a, float *smf)
{
    const int E = a.E, K = a.K, Epad = (E + 31) & ~31;
    const int TPR = max(1, 1024 / Epad), tid = threadIdx.x;
    const int slot = tid / Epad, e = tid % Epad, lane = tid & 31;
    const bool sig = a.router != COLIBRI_ROUTER_SOFTMAX;
    const int gs = sig ? E / a.n_group : E;
    float *base = smf + (long)slot * (Epad + SEL_SLOT_EXTRA);
    float *cs = base;
    float *gsc = base + Epad;
    int *kept = reinterpret_cast<int *>(base + Epad + 32);
    int *pick = reinterpret_cast<int *>(base + Epad + 64);
    float *pick_s = base + Epad + 96;
    for (int t0 = 0; t0 < a.T; t0 += TPR) {
        const int t = t0 + slot;
        const bool act = slot < TPR && t < a.T && e < E;
        const long row = (long)t * E;
        float sv = 0.0f, cv = 0.0f;
        if (act) {
            if (!sig) {
                sv = cv = a.logits[row + e];
            } else if (a.s) {
                sv = a.s[row + e];
                cv = a.c[row + e];
            } else {
                sv = (float)(1.0 / (1.0 + exp(-(double)a.logits[row + e])));
                cv = sv + (a.bias ? a.bias[e] : 0.0f);
            }
            cs[e] = cv;
        }
        __syncthreads();
        if (sig) {
            if (act && e < a.n_group) {
                // the two largest c of group e (a multiset: equal values count twice)
                float m1 = -INFINITY, m2 = -INFINITY;
                for (int i = 0; i < gs; ++i) {
                    const float v = cs[e * gs + i];
                    if (v > m1) {
                        m2 = m1;
                        m1 = v;
                    } else if (v > m2) {
                        m2 = v;
                    }
                }
                gsc[e] = gs == 1 ? m1 : m1 + m2;
            }
            __syncthreads();
            if (act && e < a.n_group) {
                const float v = gsc[e];
                int rank = 0;
                for (int g = 0; g < a.n_group; ++g)
                    rank += better(gsc[g], g, v, e) && g != e;
                kept[e] = rank < a.topk_group;
            }
            __syncthreads();
        }
        if (act && (!sig || kept[e / gs])) {
            int rank = 0;
            if (sig) {
                for (int g = 0; g < a.n_group; ++g) {
                    if (!kept[g])
                        continue;
                    for (int i = g * gs; i < (g + 1) * gs; ++i)
                        rank += better(cs[i], i, cv, e) && i != e;
                }
            } else {
                for (int i = 0; i < E; ++i)
                    rank += better(cs[i], i, cv, e) && i != e;
            }
            if (rank < K) {
                pick[rank] = e;
                pick_s[rank] = sv;
            }
        }
        __syncthreads();
        // weights: the token slot's first warp (sums in selection order on lane 0)
        if (slot < TPR && t < a.T && e < 32) {
            double m = 0.0, z = 1.0;
            if (!sig) {
                const float *l = a.logits + row;
                m = -INFINITY;
                for (int i = lane; i < E; i += 32)
                    m = fmax(m, (double)l[i]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    m = fmax(m, __shfl_xor_sync(FULL, m, o));
                z = 0.0;
                for (int i = lane; i < E; i += 32)
                    z += exp((double)l[i] - m);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    z += __shfl_xor_sync(FULL, z, o);
            }
            double p = 0.0;
            if (lane < K)
                p = sig ? (double)pick_s[lane] : exp((double)pick_s[lane] - m) / z;
            double sum = 0.0;
            for (int i = 0; i < K; ++i)
                sum += __shfl_sync(FULL, p, i);
            if (lane < K) {
                if (a.norm_topk)
                    p = p / sum;
                a.ids[(long)t * K + lane] = pick[lane];
                a.w[(long)t * K + lane] = (float)(p * (double)a.routed_scale);
            }
        }
        __syncthreads();
    }
}

size_t select_cta_smem_bytes(int E)
{
    const int Epad = (E + 31) & ~31;
    const int TPR = 1024 / Epad > 0 ? 1024 / Epad : 1;
    return (size_t)TPR * (Epad + SEL_SLOT_EXTRA) * sizeof(float);
}

// Decode (T <= 32): selection of every token with the whole CTA, then bucketing. The
// selection's shared arrays and the bucketing's counters use the same dynamic shared
// memory, one after the other.
__global__ void __launch_bounds__(1024) k_select_bucket(SelectArgs sa, BucketArgs ba)
{
    extern __shared__ int sm[];
    select_cta(sa, reinterpret_cast<float *>(sm));
    __syncthreads();  // ids in global memory are visible to the whole block
    bucket_body(ba, sm);
}

}  // namespace clb
