// Decode (T <= 32 tokens): a whole routed MoE layer in one persistent kernel: router
// logits, expert selection and bucketing, fused gate/up + SwiGLU + q8(h), down, and the
// weighted combine with the shared expert.
//
// Expert matrices are stored in row blocks of 32 rows, group-major inside a block: the 16
// bytes of one 32-column group of the block's 32 rows lie together (512 bytes), and the
// whole block is one contiguous run. A work item of an expert slot is one row block of W1
// and the same one of W3 for gate/up (one 32-group of h), or two neighbouring row blocks of
// W2 for down (64 rows of y); either way a stage holds the same group range of two 32-row
// blocks, so one code path computes both.
//
// Items are claimed from a device counter, in the order: the logit items (a block of
// router rows against a block of tokens, streamed in K-chunks), the shared expert's
// gate/up items, the routed slots' gate/up items, then the down items slot by slot. Once
// a device counter holds every logit task and every q8 group of x, each CTA selects the
// experts of every token itself (the whole CTA by rank counting, each group first ranked
// within itself, or a warp per token when the scores of all tokens do not fit), from the
// scores the logit items left in the
// workspace, buckets the pairs into its shared memory and goes on to the routed items;
// CTA 0 also writes the routing results out. CTA b's first item is item b; the counter
// hands out the rest in order. A CTA processes its items in claim order and an item waits
// only for items of lower index, each held by a running CTA (the first items all at once,
// the rest claimed earlier), so every wait below ends: routing waits for the logit items,
// a down item for the gate/up items of its slot.
//
// One CTA per SM, three roles. The producer warp claims items (two ahead, so a claim's
// latency hides behind the copies of the items before) and streams each item through a
// ring of shared-memory stages with 1-D bulk copies (a stage holds 32 group tiles of each
// of the two row blocks, with their scales: 40 KB), tagging each stage with the item and its
// position and leaving the decoded item beside it; completion is counted on a "full"
// mbarrier per stage. For a down item it
// also copies the item's rows of q8(h) into one of a few h buffers, once the gate/up
// items of its slot are done, ahead of the consumers. The consumer warps split each
// stage's groups; lane l owns row l of the block and reads its 16 bytes of a group tile
// from shared memory, so a lane accumulates whole row dots over its groups in registers.
// Each CTA quantises the activations itself (q8 of x, into shared memory). At the end of
// a chunk the consumers leave their partial sums in one of several buffers and go on; an
// epilogue warp per buffer adds them in a fixed order, writes h (SwiGLU + q8) or y, and
// publishes the result with a device-scope fence and a counter: rows of h finished per
// slot, rows of y finished per row block of d. The epilogue warp that completes a row
// block of d adds the slots' outputs for it in slot order:
// out = y_shared + sum_i w_i * y_i.
#include <mutex>

#include "kernels.cuh"

namespace clb {

namespace {

constexpr int NC = 8;                        // consumer warps
constexpr int NT = NC * 32;                  // consumer threads
constexpr int GPW = 4;                       // groups per consumer warp and stage
constexpr int SG = NC * GPW;                 // group tiles per matrix and stage
constexpr int STAGE_BYTES = 2 * SG * 640;    // 2 matrices x 32 groups x (512 + 128) bytes
constexpr int MAX_RING = 16;
constexpr size_t SMEM_BUDGET = 227 * 1024;  // the largest opt-in dynamic shared memory of a CTA
constexpr int NE_MAX = 4;                    // epilogue warps launched
constexpr int NH_MAX = 3;                    // h buffers at most
constexpr int TAG_NEW_H = 1 << 20;           // stage tag: this chunk starts a new h buffer
constexpr int TAG_END = -1, TAG_ROUTE = -2;  // stage tags (item field): end of work, routing
constexpr int LT = 8;                        // logit tasks (expert, token) per consumer warp and item
constexpr int SEL_SCRATCH = 32 * 1024;       // selection scratch of the routing CTA (bytes, at most)


__host__ __device__ constexpr int round_up(int v, int m)
{
    return (v + m - 1) / m * m;
}

struct __align__(16) DecItem {
    int mode, slot, is_shared, rb, begin, count, kdim, pad;
};

// One slot as the kernel keeps it in shared memory: its expert's matrices and its run of
// the pair list.
struct SlotInfo {
    colibri_expert ex;
    int begin, count, pad[2];
};

// A logit item: router rows [e0, e0 + ne) against tokens [t0, t0 + ntok).
struct LogitItem {
    int e0, ne, t0, ntok;
};

__device__ __forceinline__ LogitItem logit_item(const DecodeArgs &a, int idx)
{
    const int neb = (a.E + a.lg_ne - 1) / a.lg_ne;
    const int eb = idx % neb, tb = idx / neb;
    LogitItem li;
    li.e0 = eb * a.lg_ne;
    li.ne = min(a.lg_ne, a.E - li.e0);
    li.t0 = tb * a.lg_tb;
    li.ntok = min(a.lg_tb, a.T - li.t0);
    return li;
}

// What an epilogue warp needs about a finished chunk.
struct ChunkDesc {
    int mode, slot, rb, nt, pad[4];
    int orow[8];
};

// Shared memory beside the ring: see ring_layout().
struct RingLayout {
    size_t full, empty, hfull, hempty, cbar, tbar, xbar, pfull, pempty, tag, flags, ctab, desc, stab, ptab, wtab,
        act, hbuf, part, sitem, total;
    size_t hb;  // bytes of one h buffer
};

// Bytes of the routing scratch (selection and bucketing), laid over the partial-sum
// buffers (which no chunk uses before routing; the logit items keep their chains there
// too): picked ids and first-occurrence flags of the T*K pairs, then per selecting warp
// two score rows (c or logits, and s) of E floats and 32 picks.
// The selection of all T tokens at once by the whole CTA (select_cta) keeps every token's
// scores in shared memory: up to T * E = 4096.
__host__ __device__ __forceinline__ bool select_all_at_once(int T, int E)
{
    return T * E <= 4096;
}

__host__ __device__ __forceinline__ size_t route_scratch_bytes(int T, int E, int K, int sel_warps, bool select)
{
    size_t b = (8 * (size_t)T * K + 16 + 15) & ~size_t(15);
    const size_t Ep = (E + 3) & ~3;
    if (select && select_all_at_once(T, E))
        b += 2 * (size_t)T * Ep * 4 + (size_t)T * 32 * 20;  // c and s rows, group scores, kept, picks, kept list
    else if (select)
        b += (size_t)sel_warps * (8 * Ep + 128);
    return b;
}

// The x staging area: codes [TCH][d] | scales [TCH][d/32] | corrections [TCH][d/32], each
// part starting on 16 bytes.
__host__ __device__ __forceinline__ size_t x_sc_off(int d, int tch)
{
    return ((size_t)tch * d + 15) & ~size_t(15);
}
__host__ __device__ __forceinline__ size_t x_cr_off(int d, int tch)
{
    return x_sc_off(d, tch) + ((4 * (size_t)tch * (d / G) + 15) & ~size_t(15));
}
__host__ __device__ __forceinline__ size_t x_area_bytes(int d, int tch)
{
    return x_cr_off(d, tch) + ((4 * (size_t)tch * (d / G) + 15) & ~size_t(15));
}

// ring [ns][STAGE_BYTES] | full [ns] | empty [ns] | hfull [NH_MAX] | hempty [NH_MAX] |
// consumer barrier | table barrier | x barrier | pfull [NE_MAX] | pempty [NE_MAX] | stage tags [ns]
// (int2) | stage items [ns] (the producer's work item of each stage) | flags (16 B) | counters | chunk descriptors [NE_MAX] | slot table [max_slots] |
// pair list [T*K] | weights [T*K] | x staging area | h buffers [nh] (codes [TCH][fmax] |
// scales [TCH][hgs] | corrections [TCH][hgs]) | partial sums [NBUF][NC][2][TCH][32]
// (before the first chunk: the routing scratch).
__host__ __device__ __forceinline__ RingLayout ring_layout(const DecodeArgs &a, int ns, int nh, int nbuf, int tch)
{
    RingLayout L;
    const int P = a.T * a.K;
    size_t o = (size_t)ns * STAGE_BYTES;
    auto take = [&](size_t bytes, size_t align) {
        o = (o + align - 1) / align * align;
        const size_t at = o;
        o += bytes;
        return at;
    };
    L.full = take(8 * (size_t)ns, 8);
    L.empty = take(8 * (size_t)ns, 8);
    L.hfull = take(8 * NH_MAX, 8);
    L.hempty = take(8 * NH_MAX, 8);
    L.cbar = take(8, 8);
    L.tbar = take(8, 8);
    L.xbar = take(8, 8);
    L.pfull = take(8 * NE_MAX, 8);
    L.pempty = take(8 * NE_MAX, 8);
    L.tag = take(8 * (size_t)ns, 8);
    L.sitem = take(sizeof(DecItem) * (size_t)ns, 16);
    L.flags = take(16, 16);
    L.ctab = take(sizeof(Counters), 16);
    L.desc = take(sizeof(ChunkDesc) * NE_MAX, 16);
    L.stab = take(sizeof(SlotInfo) * (size_t)a.max_slots, 16);
    L.ptab = take(round_up(4 * P, 16), 16);
    L.wtab = take(round_up(4 * P, 16), 16);
    L.act = take(x_area_bytes(a.d, tch), 16);
    L.hb = round_up(tch * a.fmax + 8 * tch * a.hgs, 16);
    L.hbuf = take(L.hb * nh, 16);
    const size_t pbytes = 4 * (size_t)nbuf * NC * 2 * tch * 32;
    size_t rbytes = route_scratch_bytes(a.T, a.E, a.K, a.sel_warps, !a.ids_given);
    const size_t lbytes = 4 * (size_t)NC * LT * 32;  // logit chains
    rbytes = rbytes > lbytes ? rbytes : lbytes;
    L.part = take(pbytes > rbytes ? pbytes : rbytes, 16);  // routing scratch before the first chunk
    L.total = o;
    return L;
}

struct RingSmem {
    unsigned char *ring;
    uint64_t *full, *empty, *hfull, *hempty, *cbar, *tbar, *xbar, *pfull, *pempty;
    int2 *tag;
    DecItem *sitem;  // the work item of the stage in each ring slot, as the producer decoded it
    int *flags;  // [0] abort, [1] valid pairs, [2] distinct experts, [3] this CTA routes
    Counters *ctab;
    ChunkDesc *desc;
    SlotInfo *stab;
    int *ptab;
    float *wtab;
    unsigned char *act, *hbuf;
    size_t hb;
    float *part;
};

__device__ __forceinline__ RingSmem carve(unsigned char *sm, const DecodeArgs &a, int tch)
{
    const RingLayout L = ring_layout(a, a.ring, a.nh, a.nbuf, tch);
    RingSmem s;
    s.ring = sm;
    s.full = reinterpret_cast<uint64_t *>(sm + L.full);
    s.empty = reinterpret_cast<uint64_t *>(sm + L.empty);
    s.hfull = reinterpret_cast<uint64_t *>(sm + L.hfull);
    s.hempty = reinterpret_cast<uint64_t *>(sm + L.hempty);
    s.cbar = reinterpret_cast<uint64_t *>(sm + L.cbar);
    s.tbar = reinterpret_cast<uint64_t *>(sm + L.tbar);
    s.xbar = reinterpret_cast<uint64_t *>(sm + L.xbar);
    s.pfull = reinterpret_cast<uint64_t *>(sm + L.pfull);
    s.pempty = reinterpret_cast<uint64_t *>(sm + L.pempty);
    s.tag = reinterpret_cast<int2 *>(sm + L.tag);
    s.sitem = reinterpret_cast<DecItem *>(sm + L.sitem);
    s.flags = reinterpret_cast<int *>(sm + L.flags);
    s.ctab = reinterpret_cast<Counters *>(sm + L.ctab);
    s.desc = reinterpret_cast<ChunkDesc *>(sm + L.desc);
    s.stab = reinterpret_cast<SlotInfo *>(sm + L.stab);
    s.ptab = reinterpret_cast<int *>(sm + L.ptab);
    s.wtab = reinterpret_cast<float *>(sm + L.wtab);
    s.act = sm + L.act;
    s.hbuf = sm + L.hbuf;
    s.hb = L.hb;
    s.part = reinterpret_cast<float *>(sm + L.part);
    return s;
}

__device__ __forceinline__ void set_abort(const DecodeArgs &a, const RingSmem &s)
{
    atomicOr(a.err, ERR_WAIT_TIMEOUT);
    *reinterpret_cast<volatile int *>(s.flags) = 1;
}

__device__ __forceinline__ bool aborted(const RingSmem &s)
{
    return *reinterpret_cast<volatile int *>(s.flags) != 0;
}

// Barrier of the consumer warps on an mbarrier (count NC): bounded, unlike bar.sync, so a
// warp that gave up on a wait cannot strand the others.
__device__ __noinline__ bool consumers_sync(const RingSmem &s, uint32_t &phase, int lane)
{
    __syncwarp();
    if (lane == 0)
        mbar_arrive(s.cbar);
    const bool ok = mbar_wait(s.cbar, phase);
    phase ^= 1u;
    return ok;
}

__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Items of the shared expert's gate/up phase.
__device__ __forceinline__ int shared_gu_items(const DecodeArgs &a)
{
    return a.has_shared ? a.shared_ffn / G : 0;
}

// Work item idx of the claim order, given n_gu (one past the last gate/up item: before the
// routing table is in, the end of the shared expert's items). The logit items and the
// shared expert's items (slot 0) need nothing written by routing; the routed slots come
// from the table. The producer decodes each item once and leaves it beside each of its
// stages for the consumer warps.
__device__ __forceinline__ DecItem work_item(const DecodeArgs &a, const SlotInfo *stab, int n_gu, int idx)
{
    DecItem it{};
    if (idx < a.n_logit) {
        it.mode = MODE_LOGIT;
        it.slot = -1;
        it.kdim = a.d;
        return it;
    }
    const int sh_items = shared_gu_items(a);
    if (idx < n_gu) {
        const int r0 = idx - a.n_logit;
        it.mode = MODE_GATEUP;
        if (r0 < sh_items) {
            it.slot = 0;
            it.rb = r0;
        } else {
            const int r = r0 - sh_items, nrb = a.ffn / G;
            it.slot = (a.has_shared ? 1 : 0) + r / nrb;
            it.rb = r % nrb;
        }
    } else {
        const int r = idx - n_gu, npairs = (a.d / G + 1) / 2;
        it.mode = MODE_DOWN;
        it.slot = r / npairs;
        it.rb = 2 * (r % npairs);  // first of the two row blocks
    }
    if (a.has_shared && it.slot == 0) {
        it.is_shared = 1;
        it.begin = 0;
        it.count = a.T;
    } else {
        const SlotInfo &sl = stab[it.slot];
        it.is_shared = 0;
        it.begin = sl.begin;
        it.count = sl.count;
    }
    it.kdim = it.mode == MODE_GATEUP ? a.d : (it.is_shared ? a.shared_ffn : a.ffn);
    return it;
}

// Pair row of token c of an item's slot (the shared expert's rows follow the T*K pairs).
__device__ __forceinline__ int item_row(const DecodeArgs &a, const RingSmem &s, const DecItem &it, int c)
{
    return it.is_shared ? a.T * a.K + c : s.ptab[it.begin + c];
}

// This CTA's share of the shared expert's six parts, sent towards L2.
__device__ void prefetch_shared(const DecodeArgs &a)
{
    const size_t nib1 = (size_t)a.shared_ffn * a.d / 2, sc1 = 4 * (size_t)a.shared_ffn * (a.d / G);
    const size_t nib2 = (size_t)a.d * a.shared_ffn / 2, sc2 = 4 * (size_t)a.d * (a.shared_ffn / G);
    const void *part[6] = {a.shared.w1, a.shared.w3, a.shared.s1, a.shared.s3, a.shared.w2, a.shared.s2};
    const size_t bytes[6] = {nib1, nib1, sc1, sc1, nib2, sc2};
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        const size_t share = ((bytes[i] + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
        const size_t b0 = share * blockIdx.x;
        if (b0 >= bytes[i])
            continue;
        const size_t n = min(share, bytes[i] - b0);
        prefetch_l2(static_cast<const char *>(part[i]) + b0, (uint32_t)n);
    }
}

// (value, index) order of the selection: larger value first, then lower index.
__device__ __forceinline__ bool beats(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void top2_merge(float &m1, float &m2, float o1, float o2)
{
    // the two largest of the multiset {m1, m2, o1, o2}, given m1 >= m2 and o1 >= o2
    if (o1 > m1) {
        m2 = fmaxf(m1, o2);
        m1 = o1;
    } else {
        m2 = fmaxf(m2, o1);
    }
}

// The q8 of the tokens rows[0..nrow) of x from the workspace into the staging area, row r
// at row r: codes in even/odd word order, scales, corrections.
template <int TCH>
__device__ void stage_x_rows(const DecodeArgs &a, int8_t *codes, float *sc, int *cr, const int (&rows)[TCH], int nrow,
                             int tid)
{
    const int v16 = a.d / 16, gx = a.d / G;
    for (int i = tid; i < nrow * v16; i += NT) {
        const int r = i / v16, o = i - r * v16;
        int xr = 0;
#pragma unroll
        for (int t = 0; t < TCH; ++t)
            xr = t == r ? rows[t] : xr;
        reinterpret_cast<uint4 *>(codes + (size_t)r * a.d)[o] =
            __ldcg(reinterpret_cast<const uint4 *>(a.xq_eo + (long)xr * a.d) + o);
    }
    for (int i = tid; i < nrow * gx; i += NT) {
        const int r = i / gx, g = i - r * gx;
        int xr = 0;
#pragma unroll
        for (int t = 0; t < TCH; ++t)
            xr = t == r ? rows[t] : xr;
        cr[i] = __ldcg(a.xc + (long)xr * gx + g);
    }
    const int gs = a.d / a.group;  // scales a row
    for (int i = tid; i < nrow * gs; i += NT) {
        const int r = i / gs, g = i - r * gs;
        int xr = 0;
#pragma unroll
        for (int t = 0; t < TCH; ++t)
            xr = t == r ? rows[t] : xr;
        sc[i] = __ldcg(a.sx + (long)xr * gs + g);
    }
}

// One K-chunk of logit item idx: consumer warp w owns the item's (expert, token) tasks w,
// w + NC, ...; lane j continues the fmaf chain of its tasks over k = j, j + 32, ...
// ascending. The stage holds the chunk of the item's token rows of x ([lg_tb][lg_kc]) and
// then of its router rows ([ne][lg_kc]). The chains live in the partial-sum area (no
// chunk uses it before routing): lacc[i * 32 + lane] for task w + NC * i.
__device__ __forceinline__ void logit_chunk(const unsigned char *stg, const DecodeArgs &a, int idx, int c, float *lacc,
                                            int warp, int lane)
{
    const LogitItem li = logit_item(a, idx);
    const int kc = a.lg_kc, kcl = min(kc, a.d - c * kc);
    const float *xs = reinterpret_cast<const float *>(stg);
    const float *ws = xs + (size_t)a.lg_tb * kc;
    const int ntask = li.ne * li.ntok;
    for (int i = 0; i < LT; ++i) {
        const int task = warp + NC * i;
        if (task >= ntask)
            break;
        const int te = task / li.ntok, tt = task - te * li.ntok;
        const float *xr = xs + (size_t)tt * kc, *wr = ws + (size_t)te * kc;
        float acc = c == 0 ? 0.0f : lacc[i * 32 + lane];
        // sixteen operand pairs at a time into registers, then the sixteen fmaf of the
        // chain (the chain's order is unchanged; only the loads run ahead)
        constexpr int PF = 16;
        int k = lane;
        for (; k + 32 * (PF - 1) < kcl; k += 32 * PF) {
            float xv[PF], wv[PF];
#pragma unroll
            for (int u = 0; u < PF; ++u) {
                xv[u] = xr[k + 32 * u];
                wv[u] = wr[k + 32 * u];
            }
#pragma unroll
            for (int u = 0; u < PF; ++u)
                acc = fmaf(xv[u], wv[u], acc);
        }
        for (; k < kcl; k += 32)
            acc = fmaf(xr[k], wr[k], acc);
        lacc[i * 32 + lane] = acc;
    }
}

// The end of logit item idx: each task's 32 chains joined by a butterfly (offsets 16, 8,
// 4, 2, 1: every lane then holds the halving tree's sum); lane i writes task w + NC * i:
// the logit and, in sigmoid mode, s = fp32(sigmoid(l)) evaluated in fp64 and c = s + bias.
// Returns the tasks written by this warp.
__device__ __forceinline__ int logit_finish(const DecodeArgs &a, int idx, const float *lacc, int warp, int lane)
{
    const LogitItem li = logit_item(a, idx);
    const int ntask = li.ne * li.ntok;
    float mine = 0.0f;
    int nw = 0;
    for (int i = 0; i < LT; ++i) {
        const int task = warp + NC * i;
        if (task >= ntask)
            break;
        float v = lacc[i * 32 + lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            v = v + __shfl_xor_sync(FULL, v, o);
        mine = lane == i ? v : mine;
        ++nw;
    }
    if (lane < nw) {
        const int task = warp + NC * lane;
        const int te = task / li.ntok, tt = task - te * li.ntok;
        const int e = li.e0 + te;
        const long o = (long)(li.t0 + tt) * a.E + e;
        a.logits[o] = mine;
        if (a.router != COLIBRI_ROUTER_SOFTMAX) {
            const float sv = (float)(1.0 / (1.0 + exp(-(double)mine)));
            a.rs[o] = sv;
            a.rc[o] = sv + (a.bias ? a.bias[e] : 0.0f);
        }
    }
    return nw;
}

// Expert selection of token t by one warp, from the router scores in the workspace (cs,
// ss: this warp's scratch of E floats each; pick: 32 ints). Sigmoid mode: lane g takes
// the two largest biased scores c of group g, their sum is the group score, and the
// topk_group best groups are kept (ties: lower group index); then every allowed expert
// counts the allowed experts that beat it by (c, lower index), and the one that exactly
// k others beat is the k-th pick: the same ids, in the same order, as a sequential
// selection. w = s / sum(s) * routed_scale with a compensated fp32 sum in selection order.
// Softmax mode: top_k by logit, w = softmax over all experts in fp64. Writes the ids and
// weights to sids and wtab (shared memory); the writer CTA also to the caller's ids and w.
__device__ void select_warp(const DecodeArgs &a, int t, float *cs, float *ss, int *pick, int *sids, float *wtab,
                            bool writer, int lane)
{
    const int E = a.E, K = a.K;
    const bool sig = a.router != COLIBRI_ROUTER_SOFTMAX;
    const int NG = sig ? a.n_group : 1, gs = E / NG;
    const long base = (long)t * E;
    __syncwarp();
    for (int e0 = 0; e0 < E; e0 += 32 * 8) {
        // eight loads of each row in flight at once
        float cv[8], sv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + 32 * u + lane;
            cv[u] = e < E ? rank_score(__ldcg((sig ? a.rc : a.logits) + base + e)) : 0.0f;
            sv[u] = sig && e < E ? __ldcg(a.rs + base + e) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + 32 * u + lane;
            if (e < E) {
                cs[e] = cv[u];
                ss[e] = sv[u];
            }
        }
    }
    __syncwarp();
    unsigned kept = 1u;
    if (sig) {
        float gsc = -INFINITY;  // lane g: the score of group g
        if (lane < NG) {
            float m1 = -INFINITY, m2 = -INFINITY;
            for (int j = lane * gs; j < (lane + 1) * gs; ++j)
                top2_merge(m1, m2, cs[j], -INFINITY);
            gsc = gs == 1 ? m1 : m1 + m2;
        }
        int rank = 0;
        for (int h = 0; h < NG; ++h)
            rank += beats(__shfl_sync(FULL, gsc, h), h, gsc, lane);
        kept = __ballot_sync(FULL, lane < NG && rank < a.topk_group);
    }
    const bool vec = (gs & 3) == 0;
    for (int e = lane; e < E; e += 32) {
        if (!((kept >> (e / gs)) & 1u))
            continue;
        const float v = cs[e];
        int r = 0;
        for (int g = 0; g < NG; ++g) {
            if (!((kept >> g) & 1u))
                continue;
            if (vec) {
                const float4 *q4 = reinterpret_cast<const float4 *>(cs + g * gs);
                int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
                for (int j = 0; j < gs / 4; ++j) {
                    const float4 x = q4[j];
                    const int f = g * gs + 4 * j;
                    r0 += beats(x.x, f, v, e);
                    r1 += beats(x.y, f + 1, v, e);
                    r2 += beats(x.z, f + 2, v, e);
                    r3 += beats(x.w, f + 3, v, e);
                }
                r += r0 + r1 + r2 + r3;
            } else {
                for (int f = g * gs; f < (g + 1) * gs; ++f)
                    r += beats(cs[f], f, v, e);
            }
        }
        if (r < K)
            pick[r] = e;
    }
    __syncwarp();
    const bool have = lane < K;
    const int my_id = have ? pick[lane] : 0;
    float wt = 0.0f;
    if (sig) {
        // compensated (TwoSum) sum of the k scores in selection order, one division
        const float sv = have ? ss[my_id] : 0.0f;
        float hi = 0.0f, lo = 0.0f;
        for (int i = 0; i < K; ++i) {
            const float x = __shfl_sync(FULL, sv, i);
            const float u = hi + x, bb = u - hi;
            lo += (hi - (u - bb)) + (x - bb);
            hi = u;
        }
        const float sum = hi + lo;
        wt = (a.norm_topk ? __fdiv_rn(sv, sum) : sv) * a.routed_scale;
    } else {
        double m = -INFINITY;
        for (int i = lane; i < E; i += 32)
            m = fmax(m, (double)cs[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = fmax(m, __shfl_xor_sync(FULL, m, o));
        double z = 0.0;
        for (int i = lane; i < E; i += 32)
            z += exp((double)cs[i] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            z += __shfl_xor_sync(FULL, z, o);
        double p = have ? exp((double)cs[my_id] - m) / z : 0.0;
        double sum = 0.0;
        for (int i = 0; i < K; ++i)
            sum += __shfl_sync(FULL, p, i);
        if (a.norm_topk)
            p = p / sum;
        wt = (float)(p * (double)a.routed_scale);
    }
    if (have) {
        sids[t * K + lane] = my_id;
        wtab[t * K + lane] = wt;
        if (writer) {
            a.ids[(long)t * K + lane] = my_id;
            a.w_out[(long)t * K + lane] = wt;
        }
    }
}

// Expert selection for the T tokens by the consumer warps, in shared memory (every CTA
// the same way). The k-th pick of the sequential selection (repeatedly take the best
// remaining candidate) is the candidate that exactly k others beat, so each candidate
// counts the allowed candidates that beat it and, if that rank is below top_k, takes
// position rank; groups are kept the same way. Sigmoid mode: group score = sum of the
// group's two largest biased scores c, top topk_group groups, top_k by c inside them,
// w = s / sum(s) * routed_scale with a compensated fp32 sum in selection order. Softmax
// mode: top_k by logit, w = softmax over all experts (fp32, compensated). Writes the ids
// and weights to sids and s.wtab; the writer CTA also to the caller's ids and w. Used when
// the scores of all T tokens fit the scratch (T * E <= 4096); select_warp otherwise.
//
// Chunked form (groups of at most 32 experts in sigmoid mode, runs of 32 experts in softmax
// mode, when the kept chunks' best kk = min(top_k, chunk) fit one warp): one warp a (token,
// chunk) ranks the chunk's experts among themselves, one lane an expert, and lists its kk
// best in order (the two best give the group score); then one warp a token ranks the
// listed experts of its kept chunks among themselves. Every expert of the overall top_k is
// among the kk best of its own chunk under the same order, so the picks are the same as
// ranking every allowed expert against every other, at a quarter of the comparisons or
// less.
__device__ bool select_cta(const DecodeArgs &a, const RingSmem &s, float *scr, int *sids, bool writer, uint32_t &cph,
                           int tid, int warp, int lane)
{
    const int E = a.E, K = a.K, T = a.T;
    const bool sig = a.router != COLIBRI_ROUTER_SOFTMAX;
    const int NG = sig ? a.n_group : 1, gs = E / NG;
    const int Ep = (E + 3) & ~3;
    float *cs = scr;                   // c (sigmoid) or logits [T][Ep]
    float *ss = cs + (size_t)T * Ep;   // s [T][Ep] (sigmoid)
    float *gsc = ss + (size_t)T * Ep;  // group scores [T][32]
    int *kept = reinterpret_cast<int *>(gsc + (size_t)T * 32);
    int *pick = kept + (size_t)T * 32;
    float *ps = reinterpret_cast<float *>(pick + (size_t)T * 32);
    for (int i = tid; i < T * E; i += NT) {
        const int t = i / E, e = i - t * E;
        cs[t * Ep + e] = rank_score(sig ? __ldcg(a.rc + i) : __ldcg(a.logits + i));
        if (sig)
            ss[t * Ep + e] = __ldcg(a.rs + i);
    }
    named_sync(1, NT);
    // chunks: the groups (sigmoid) or runs of 32 experts (softmax); kk best listed a chunk
    const int cl = sig ? gs : min(E, 32), nch = (E + cl - 1) / cl, kk = min(K, cl);
    const int nkept = sig ? a.topk_group : nch;
    const bool chunked = cl <= 32 && nch <= 32 && nch * kk <= 64 && nkept * kk <= 32;
    int16_t *ctop = reinterpret_cast<int16_t *>(ps + (size_t)T * 32);  // [T][64]: chunk ch at ch * kk
    if (chunked) {
        for (int i = warp; i < T * nch; i += NC) {
            const int t = i / nch, ch = i - t * nch;
            const int base = ch * cl, len = min(cl, E - base);
            const float *row = cs + (size_t)t * Ep + base;
            const bool live = lane < len;
            const float v = live ? row[lane] : -INFINITY;
            int r = 0;  // the chunk's experts that beat this lane's
            if (len == 32) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(row + j);
                    r += (x.x > v || (x.x == v && j < lane)) + (x.y > v || (x.y == v && j + 1 < lane)) +
                         (x.z > v || (x.z == v && j + 2 < lane)) + (x.w > v || (x.w == v && j + 3 < lane));
                }
            } else {
                for (int j = 0; j < len; ++j) {
                    const float x = row[j];
                    r += x > v || (x == v && j < lane);
                }
            }
            if (live && r < kk)
                ctop[t * 64 + ch * kk + r] = (int16_t)(base + lane);
            if (sig) {
                const unsigned m0 = __ballot_sync(FULL, live && r == 0), m1 = __ballot_sync(FULL, live && r == 1);
                const float v0 = __shfl_sync(FULL, v, __ffs(m0) - 1);
                const float v1 = __shfl_sync(FULL, v, m1 ? __ffs(m1) - 1 : 0);
                if (lane == 0)
                    gsc[t * 32 + ch] = len == 1 ? v0 : v0 + v1;
            }
        }
        named_sync(1, NT);
    }
    if (!chunked && sig) {
        for (int i = warp; i < T * NG; i += NC) {
            const int t = i / NG, g = i - t * NG;
            const float *row = cs + (size_t)t * Ep + g * gs;
            float m1 = -INFINITY, m2 = -INFINITY;
            for (int j = lane; j < gs; j += 32)
                top2_merge(m1, m2, row[j], -INFINITY);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float o1 = __shfl_xor_sync(FULL, m1, o), o2 = __shfl_xor_sync(FULL, m2, o);
                top2_merge(m1, m2, o1, o2);
            }
            if (lane == 0)
                gsc[t * 32 + g] = gs == 1 ? m1 : m1 + m2;
        }
        named_sync(1, NT);
        for (int i = tid; i < T * NG; i += NT) {
            const int t = i / NG, g = i - t * NG;
            const float v = gsc[t * 32 + g];
            int rank = 0;
            for (int h = 0; h < NG; ++h)
                rank += beats(gsc[t * 32 + h], h, v, g);
            kept[t * 32 + g] = rank < a.topk_group;
        }
        named_sync(1, NT);
    }
    // rank of each allowed candidate, one thread a candidate: the allowed candidates of its
    // token that beat it, counted as those with a larger c plus those with an equal c and a
    // lower index, over the kept groups listed in shared memory
    int *klist = reinterpret_cast<int *>(ps + (size_t)T * 32);  // [T][32] kept group ids
    if (!chunked && sig) {
        for (int t = warp; t < T; t += NC) {
            const bool k = lane < NG && kept[t * 32 + lane];
            const unsigned m = __ballot_sync(FULL, k);
            if (k)
                klist[t * 32 + __popc(m & ((1u << lane) - 1))] = lane;
        }
        named_sync(1, NT);
    }
    const int nk = sig ? a.topk_group : 1;
    for (int i = chunked ? T * E : tid; i < T * E; i += NT) {
        const int t = i / E, e = i - t * E;
        if (sig && !kept[t * 32 + e / gs])
            continue;
        const float *row = cs + (size_t)t * Ep;
        const float v = row[e];
        int gt = 0, eq = 0;
        for (int kk = 0; kk < nk; ++kk) {
            const int j0 = (sig ? klist[t * 32 + kk] : 0) * gs, j1 = j0 + gs;
            int j = j0;
            if ((gs & 7) == 0) {
                for (; j < j1; j += 8) {
                    const float4 x0 = *reinterpret_cast<const float4 *>(row + j);
                    const float4 x1 = *reinterpret_cast<const float4 *>(row + j + 4);
                    gt += (x0.x > v) + (x0.y > v) + (x0.z > v) + (x0.w > v) + (x1.x > v) + (x1.y > v) + (x1.z > v) +
                          (x1.w > v);
                    eq += (x0.x == v && j < e) + (x0.y == v && j + 1 < e) + (x0.z == v && j + 2 < e) +
                          (x0.w == v && j + 3 < e) + (x1.x == v && j + 4 < e) + (x1.y == v && j + 5 < e) +
                          (x1.z == v && j + 6 < e) + (x1.w == v && j + 7 < e);
                }
            }
            for (; j < j1; ++j) {
                const float x = row[j];
                gt += x > v;
                eq += x == v && j < e;
            }
        }
        const int rank = gt + eq;
        if (rank < K) {
            pick[t * 32 + rank] = e;
            ps[t * 32 + rank] = sig ? ss[t * Ep + e] : cs[t * Ep + e];
        }
    }
    if (!chunked)
        named_sync(1, NT);
    for (int t = warp; t < T; t += NC) {
        if (chunked) {
            // the kept chunks (ascending), then lane q * kk + r holds the r-th best of the
            // q-th kept chunk and counts the listed experts that beat it
            unsigned kmask;
            if (sig) {
                const float gv = lane < nch ? gsc[t * 32 + lane] : 0.0f;
                int rk = 0;
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                    const float x = __shfl_sync(FULL, gv, h);
                    rk += h < nch && beats(x, h, gv, lane);
                }
                kmask = __ballot_sync(FULL, lane < nch && rk < a.topk_group);
            } else {
                kmask = nch == 32 ? FULL : (1u << nch) - 1u;
            }
            const int q = lane / kk, r = lane - q * kk;
            unsigned mm = kmask;
            for (int z = 0; z < q && mm; ++z)
                mm &= mm - 1u;
            int e = -1;
            if (lane < nkept * kk && mm) {
                const int ch = __ffs(mm) - 1;
                if (r < min(kk, E - ch * cl))
                    e = ctop[t * 64 + ch * kk + r];
            }
            const bool valid = e >= 0;
            const float v = valid ? cs[(size_t)t * Ep + e] : -INFINITY;
            const unsigned vm = __ballot_sync(FULL, valid);
            int rank = 0;  // lanes without a candidate are outside vm
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float xv = __shfl_sync(FULL, v, c);
                const int xe = __shfl_sync(FULL, e, c);
                rank += ((vm >> c) & 1u) && beats(xv, xe, v, e);
            }
            if (valid && rank < K) {
                pick[t * 32 + rank] = e;
                ps[t * 32 + rank] = sig ? ss[(size_t)t * Ep + e] : v;
            }
            __syncwarp();
        }
        float wt = 0.0f;
        if (sig) {
            // compensated (TwoSum) sum of the k scores in selection order, one division
            const float sv = lane < K ? ps[t * 32 + lane] : 0.0f;
            float hi = 0.0f, lo = 0.0f;
            for (int i = 0; i < K; ++i) {
                const float x = __shfl_sync(FULL, sv, i);
                const float u = hi + x, bb = u - hi;
                lo += (hi - (u - bb)) + (x - bb);
                hi = u;
            }
            const float sum = hi + lo;
            wt = (a.norm_topk ? __fdiv_rn(sv, sum) : sv) * a.routed_scale;
        } else {
            // softmax weights in fp32, within a few 1e-7 of the fp64 definition: each
            // exp(l - m) takes the argument's rounding error back to first order (the error
            // of l - m is exact by TwoSum), expf errs by at most 2 ulp, and the sums over
            // the experts and the picks are compensated (fp64 exp on this part's small fp64
            // rate took several microseconds per token)
            const float *l = cs + (size_t)t * Ep;
            float m = -INFINITY;
            for (int i = lane; i < E; i += 32)
                m = fmaxf(m, l[i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
            auto ex = [&](float x) {
                const float d = x - m, bb = d - x;
                const float err = (x - (d - bb)) + (-m - bb);  // d + err == x - m exactly
                const float e = expf(d);
                return fmaf(e, err, e);
            };
            auto add2 = [](float &hi, float &lo, float x) {  // TwoSum accumulate
                const float u = hi + x, bb = u - hi;
                lo += (hi - (u - bb)) + (x - bb);
                hi = u;
            };
            float zh = 0.0f, zl = 0.0f;
            for (int i = lane; i < E; i += 32)
                add2(zh, zl, ex(l[i]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float oh = __shfl_xor_sync(FULL, zh, o), ol = __shfl_xor_sync(FULL, zl, o);
                add2(zh, zl, oh);
                zl += ol;
            }
            const float z = zh + zl;
            float p = lane < K ? __fdiv_rn(ex(ps[t * 32 + lane]), z) : 0.0f;
            if (a.norm_topk) {
                float sh = 0.0f, sl = 0.0f;
                for (int i = 0; i < K; ++i)
                    add2(sh, sl, __shfl_sync(FULL, p, i));
                p = __fdiv_rn(p, sh + sl);
            }
            wt = p * a.routed_scale;
        }
        if (lane < K) {
            const int id = pick[t * 32 + lane];
            sids[t * K + lane] = id;
            s.wtab[t * K + lane] = wt;
            if (writer) {
                a.ids[(long)t * K + lane] = id;
                a.w_out[(long)t * K + lane] = wt;
            }
        }
    }
    return true;
}

// The shared expert's slot (0) and the counters, from the valid pairs and the distinct
// routed experts, into shared memory (and the workspace, by the writer CTA).
__device__ __forceinline__ void write_counters(const DecodeArgs &a, const RingSmem &s, bool writer, int n_valid,
                                               int n_routed)
{
    const int sbase = a.has_shared ? 1 : 0;
    if (a.has_shared) {
        SlotInfo si;
        si.ex = a.shared;
        si.begin = 0;
        si.count = a.T;
        si.pad[0] = si.pad[1] = 0;
        s.stab[0] = si;
        if (writer) {
            Slot sl;
            sl.expert = -1;
            sl.begin = 0;
            sl.count = a.T;
            sl.pad = 0;
            a.slots[0] = sl;
        }
    }
    Counters ct;
    ct.n_slots = sbase + n_routed;
    ct.n_routed = n_routed;
    ct.n_items_gateup = shared_gu_items(a) + n_routed * (a.ffn / G);
    ct.n_items_down = ct.n_slots * ((a.d / G + 1) / 2);
    ct.n_rows = n_valid + (a.has_shared ? a.T : 0);
    ct.pad[0] = ct.pad[1] = ct.pad[2] = 0;
    *s.ctab = ct;
    if (writer)
        *a.counters = ct;
}

// Bucketing of at most 32 pairs by one warp (lane p holds pair p): pair list stable by
// expert, slots = the shared expert then the distinct valid experts in ascending id,
// counters, into shared memory; the writer CTA also writes them, with the bucket
// offsets, to the workspace and flags bad ids (outside [0, E), or twice in a token).
__device__ void bucket_warp(const DecodeArgs &a, const RingSmem &s, const int *sids, bool writer, int lane)
{
    const int T = a.T, K = a.K, E = a.E, P = T * K;
    const int sbase = a.has_shared ? 1 : 0;
    __syncwarp();
    const bool live = lane < P;
    const int e = live ? sids[lane] : -1;
    const bool valid = live && e >= 0 && e < E;
    // lanes holding the same id (lanes past P get keys of their own)
    const unsigned same = __match_any_sync(FULL, live ? e : -2 - lane);
    const unsigned below = (1u << lane) - 1u;
    const int tok0 = live ? lane - lane % K : 0;
    const unsigned in_tok = below & ~((1u << tok0) - 1u);
    const bool dup = live && (same & in_tok) != 0;
    const bool fst = valid && (same & below) == 0;
    if (writer && live && (!valid || dup))
        atomicOr(a.err, ERR_BAD_ID);
    colibri_expert ex{};
    if (fst)
        ex = a.experts[e];  // in flight during the counting below
    const unsigned fmask = __ballot_sync(FULL, fst);
    const int n_valid = __popc(__ballot_sync(FULL, valid)), n_routed = __popc(fmask);
    int less = 0, dless = 0;
    for (int j = 0; j < P; ++j) {
        const int ej = __shfl_sync(FULL, e, j);
        const bool vj = ej >= 0 && ej < E;
        less += vj && ej < e;
        dless += ((fmask >> j) & 1) && ej < e;
    }
    if (valid) {
        const int pos = __popc(same & below);
        s.ptab[less + pos] = lane;
        if (writer)
            a.pairs[less + pos] = lane;
        if (fst) {
            SlotInfo si;
            si.ex = ex;
            si.begin = less;
            si.count = __popc(same);
            si.pad[0] = si.pad[1] = 0;
            s.stab[sbase + dless] = si;
            if (writer) {
                Slot sl;
                sl.expert = e;
                sl.begin = less;
                sl.count = si.count;
                sl.pad = 0;
                a.slots[sbase + dless] = sl;
            }
        }
    }
    if (writer) {
        for (int x = lane; x <= E; x += 32) {
            int c = 0;
            for (int q = 0; q < P; ++q)
                c += sids[q] >= 0 && sids[q] < x;
            a.offsets[x] = c;
        }
    }
    if (lane == 0)
        write_counters(a, s, writer, n_valid, n_routed);
}

// The same for more than 32 pairs, by all consumer threads (O(P^2) comparisons, P <=
// 1024), with first-occurrence flags in shared memory.
__device__ bool bucket_cta(const DecodeArgs &a, const RingSmem &s, const int *sids, int *first, bool writer,
                           uint32_t &cph, int tid, int lane)
{
    const int T = a.T, K = a.K, E = a.E, P = T * K;
    // whole warps take the pairs (lane l pair p0 + l), so the two counts go in with one
    // shared-memory atomic per warp
    for (int p0 = tid & ~31; p0 < P; p0 += NT) {
        const int p = p0 + lane;
        const bool live = p < P;
        const int e = live ? sids[p] : -1;
        const bool valid = live && e >= 0 && e < E;
        bool dup = false, fst = valid;
        if (live) {
            const int tok0 = p - p % K;
            int q = 0;
            if ((P & 3) == 0) {
                for (; q + 4 <= p; q += 4) {
                    const int4 e4 = *reinterpret_cast<const int4 *>(sids + q);
                    const bool s0 = e4.x == e, s1 = e4.y == e, s2 = e4.z == e, s3 = e4.w == e;
                    dup |= (s0 && q >= tok0) || (s1 && q + 1 >= tok0) || (s2 && q + 2 >= tok0) ||
                           (s3 && q + 3 >= tok0);
                    fst &= !(s0 || s1 || s2 || s3);
                }
            }
            for (; q < p; ++q) {
                const bool same = sids[q] == e;
                dup |= same && q >= tok0;
                fst &= !same;
            }
            if (writer && (!valid || dup))
                atomicOr(a.err, ERR_BAD_ID);
            first[p] = fst;
        }
        const int nv = __popc(__ballot_sync(FULL, valid)), nf = __popc(__ballot_sync(FULL, fst));
        if (lane == 0) {
            if (nv)
                atomicAdd(&s.flags[1], nv);
            if (nf)
                atomicAdd(&s.flags[2], nf);
        }
    }
    named_sync(1, NT);
    const int sbase = a.has_shared ? 1 : 0;
    // four pairs a 16-byte load when the two arrays allow it (P a multiple of 4)
    const int P4 = (P & 3) == 0 ? P : 0;
    for (int p = tid; p < P; p += NT) {
        const int e = sids[p];
        if (e < 0 || e >= E)
            continue;
        const bool fst = first[p];
        colibri_expert ex{};
        if (fst)
            ex = a.experts[e];  // in flight during the counting below
        int less = 0, pos = 0, cnt = 0, dless = 0;
        auto count = [&](int q, int eq, int fq) {
            const bool v = eq >= 0 && eq < E;
            less += v && eq < e;
            pos += q < p && eq == e;
            cnt += eq == e;
            dless += fq && eq < e;
        };
        for (int q = 0; q < P4; q += 4) {
            const int4 e4 = *reinterpret_cast<const int4 *>(sids + q);
            const int4 f4 = *reinterpret_cast<const int4 *>(first + q);
            count(q, e4.x, f4.x);
            count(q + 1, e4.y, f4.y);
            count(q + 2, e4.z, f4.z);
            count(q + 3, e4.w, f4.w);
        }
        for (int q = P4; q < P; ++q)
            count(q, sids[q], first[q]);
        s.ptab[less + pos] = p;
        if (writer)
            a.pairs[less + pos] = p;
        if (fst) {
            SlotInfo si;
            si.ex = ex;
            si.begin = less;
            si.count = cnt;
            si.pad[0] = si.pad[1] = 0;
            s.stab[sbase + dless] = si;
            if (writer) {
                Slot sl;
                sl.expert = e;
                sl.begin = less;
                sl.count = cnt;
                sl.pad = 0;
                a.slots[sbase + dless] = sl;
            }
        }
    }
    if (writer) {
        for (int e = tid; e <= E; e += NT) {
            int less = 0;
            for (int q = 0; q < P; ++q)
                less += sids[q] >= 0 && sids[q] < e;
            a.offsets[e] = less;
        }
    }
    if (tid == 0)
        write_counters(a, s, writer, s.flags[1], s.flags[2]);
    return true;
}

// Routing of this CTA, at its routing stage: once every logit task of the layer is in
// (a device counter), every token's selection (or the given ids and weights), then
// bucketing, into shared memory; CTA 0 also writes the results to the workspace and the
// caller's ids and w. Then the producer may read the table (tbar). The consumer warps
// meet on hardware barrier 1 here: every one of them runs this code to its end (the only
// wait, for the counter, is bounded and taken by one thread before the first barrier).
__device__ bool route_cta(const DecodeArgs &a, const RingSmem &s, uint32_t &cph, int tid, int warp, int lane)
{
    const int T = a.T, K = a.K, P = T * K;
    const bool writer = blockIdx.x == 0;
    // all T tokens' x codes staged at once, by bulk copies when the parts are whole 16-byte
    // runs
    const bool x_all = T <= a.tch, x_bulk = x_all && ((long)T * a.d) % (4 * a.group) == 0;
    int *sids = reinterpret_cast<int *>(s.part);
    int *first = sids + P;
    unsigned char *scr0 = reinterpret_cast<unsigned char *>(s.part) + ((8 * (size_t)P + 16 + 15) & ~size_t(15));
    const int Ep = (a.E + 3) & ~3;
    if (tid == 0) {
        s.flags[1] = s.flags[2] = 0;
        int ok = 1;
        // every logit task and every q8 group of x of the layer
        ok = wait_count_geq(a.route_done, (a.ids_given ? 0 : a.E * a.T) + a.T * (a.d / a.group));
        __threadfence();
        if (ok && x_bulk) {
            // the q8 of all T tokens into the x staging area (codes in even/odd order,
            // scales, corrections)
            fence_proxy_async_global();
            const uint32_t nc = (uint32_t)(a.T * a.d), ns = (uint32_t)(4 * a.T * (a.d / a.group)),
                           nr = (uint32_t)(4 * a.T * (a.d / G));
            unsigned char *act = reinterpret_cast<unsigned char *>(s.act);
            mbar_arrive_expect_tx(s.xbar, nc + ns + nr);
            bulk_g2s(act, a.xq_eo, nc, s.xbar);
            bulk_g2s(act + x_sc_off(a.d, a.tch), a.sx, ns, s.xbar);
            bulk_g2s(act + x_cr_off(a.d, a.tch), a.xc, nr, s.xbar);
        }
        s.flags[3] = ok;
    }
    named_sync(1, NT);
    if (!s.flags[3]) {
        if (lane == 0)
            set_abort(a, s);
        return false;
    }
    if (a.ids_given) {
        for (int i = tid; i < P; i += NT) {
            sids[i] = __ldcg(a.ids + i);
            s.wtab[i] = __ldcg(a.w_in + i);
        }
    } else if (select_all_at_once(T, a.E)) {
        if (!select_cta(a, s, reinterpret_cast<float *>(scr0), sids, writer, cph, tid, warp, lane))
            return false;
    } else if (warp < a.sel_warps) {
        float *cs = reinterpret_cast<float *>(scr0 + (size_t)warp * (8 * Ep + 128));
        int *pick = reinterpret_cast<int *>(cs + 2 * Ep);
        for (int t = warp; t < T; t += a.sel_warps)
            select_warp(a, t, cs, cs + Ep, pick, sids, s.wtab, writer, lane);
    }
    named_sync(1, NT);
    if (P <= 32) {
        if (warp == 0)
            bucket_warp(a, s, sids, writer, lane);
    } else if (!bucket_cta(a, s, sids, first, writer, cph, tid, lane)) {
        return false;
    }
    named_sync(1, NT);
    if (tid == 0)
        mbar_arrive(s.tbar);  // the producer may read the table
    // the staged q8 of x before the first gate/up stage
    if (x_bulk && !mbar_wait(s.xbar, 0)) {
        if (lane == 0)
            set_abort(a, s);
        return false;
    }
    if (x_all && !x_bulk) {
        const int v16 = a.d / 16, gx = a.d / G;
        int8_t *codes = reinterpret_cast<int8_t *>(s.act);
        float *sc = reinterpret_cast<float *>(s.act + x_sc_off(a.d, a.tch));
        int *cr = reinterpret_cast<int *>(s.act + x_cr_off(a.d, a.tch));
        for (int i = tid; i < T * v16; i += NT)
            reinterpret_cast<uint4 *>(codes)[i] = __ldcg(reinterpret_cast<const uint4 *>(a.xq_eo) + i);
        for (int i = tid; i < T * gx; i += NT)
            cr[i] = __ldcg(a.xc + i);
        for (int i = tid; i < T * (a.d / a.group); i += NT)
            sc[i] = __ldcg(a.sx + i);
        named_sync(1, NT);
    }
    return true;
}

// Partial dots of one stage: consumer warp w takes 32-column tiles w, w + NC, ... of the
// stage. Activation row t of the chunk sits at row rows[t] of the staged codes (row stride
// cstride bytes), corrections (gstride a row, one per 32 columns) and scales (sstride a
// row, one per group: tile g >> gsh, gsh = 1 for 64-element groups). The stage holds one
// weight scale tile per group.
template <int TCH>
__device__ __forceinline__ void consume(const unsigned char *stg, const int8_t *codes, const float *sc,
                                        const int *corr, int cstride, int gstride, int sstride, int gsh,
                                        const int (&rows)[TCH], int ng, int g0, int nt, int warp, int lane,
                                        float (&acc)[2][TCH])
{
    constexpr int M = 2;
    constexpr int scale_off = M * SG * 512;
    const int n = min(SG, ng - g0);
    if (n == SG) {
        // a full stage (every stage but an item's ragged last one): the warp's weight words
        // and scales of all its tiles are loaded up front, so that the dot chains of the
        // tiles overlap instead of running one tile after the other; the sums per (m, t)
        // still run over the tiles in ascending order
        uint4 wv[GPW][M];
        float sw[GPW][M];
#pragma unroll
        for (int u = 0; u < GPW; ++u) {
            const int j = warp + u * NC;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                wv[u][m] = *reinterpret_cast<const uint4 *>(stg + (m * SG + j) * 512 + lane * 16);
                sw[u][m] = *reinterpret_cast<const float *>(stg + scale_off + (m * SG + (j >> gsh)) * 128 + lane * 4);
            }
        }
#pragma unroll
        for (int t = 0; t < TCH; ++t) {
            if (t < nt) {
                const int r = rows[t];
#pragma unroll
                for (int u = 0; u < GPW; ++u) {
                    const int g = g0 + warp + u * NC;
                    const uint4 *xa = reinterpret_cast<const uint4 *>(codes + (size_t)r * cstride + g * G);
                    const uint4 A0 = xa[0], A1 = xa[1];
                    const int cr = corr[r * gstride + g];
                    const float sa = sc[r * sstride + (g >> gsh)];
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const int D = dot_split(split_nibbles(wv[u][m]), A0, A1, cr);
                        acc[m][t] = fmaf((float)D, sw[u][m] * sa, acc[m][t]);
                    }
                }
            }
        }
        return;
    }
#pragma unroll
    for (int u = 0; u < GPW; ++u) {
        const int j = warp + u * NC;
        if (j < n) {
            const int g = g0 + j;
            NibbleSplit nsp[M];
            float sw[M];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                nsp[m] = split_nibbles(*reinterpret_cast<const uint4 *>(stg + (m * SG + j) * 512 + lane * 16));
                sw[m] = *reinterpret_cast<const float *>(stg + scale_off + (m * SG + (j >> gsh)) * 128 + lane * 4);
            }
#pragma unroll
            for (int t = 0; t < TCH; ++t) {
                if (t < nt) {
                    const int r = rows[t];
                    const uint4 *xa = reinterpret_cast<const uint4 *>(codes + (size_t)r * cstride + g * G);
                    const uint4 A0 = xa[0], A1 = xa[1];
                    const int cr = corr[r * gstride + g];
                    const float sa = sc[r * sstride + (g >> gsh)];
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const int D = dot_split(nsp[m], A0, A1, cr);
                        acc[m][t] = fmaf((float)D, sw[m] * sa, acc[m][t]);
                    }
                }
            }
        }
    }
}

// ---------------- producer (one thread) ----------------
template <int TCH>
__device__ void run_producer(const DecodeArgs &a, const RingSmem &s)
{
    const int NS = a.ring, NH = a.nh;
    if (blockIdx.x == 0)
        prefetch_l2(a.experts, (uint32_t)(((size_t)a.E * sizeof(colibri_expert) + 15) & ~size_t(15)));
    grid_dep_wait();  // inputs and the zeroed counters are in
    const uint64_t pol = policy_evict_first();
    const int gsh = a.group == 64 ? 1 : 0;           // 32-column tile -> group
    const int pre = a.n_logit + shared_gu_items(a);  // items that need no routing table
    int n_gu = pre, total = 0x7fffffff;              // until the table is in
    bool have_table = false, route_posted = false;
    uint32_t st = 0, hsw = 0;  // stages posted, h buffers filled
    int hslot = -1, hch = -1;  // rows in the newest h buffer
    uint64_t h_ready = 0;      // slots (below 64) whose rows of h are all published
    // the ring slot of stage st, once the consumers have released it; the slot and the
    // lap parity are kept incrementally (no division on this path)
    uint32_t pslot = 0, plap = 0;
    auto acquire = [&](uint32_t &slot) -> bool {
        slot = pslot;
        if (st >= (uint32_t)NS && !mbar_wait(&s.empty[slot], plap ^ 1u)) {
            set_abort(a, s);
            return false;
        }
        if (++pslot == (uint32_t)NS) {
            pslot = 0;
            plap ^= 1u;
        }
        return !aborted(s);
    };
    // claims run two items ahead of the item being streamed, except behind a logit item:
    // the next claim waits until the logit item's bytes have landed, so that the logit
    // items (claimed first) spread over all CTAs instead of pairing up. Each CTA's first
    // item is its own index (no counter round trip before the first copy); the counter
    // hands out the items from gridDim.x on, in order
    auto claim = [&]() { return (int)gridDim.x + atomicAdd(a.claim, 1); };
    int idx = blockIdx.x, ahead = idx < a.n_logit ? -1 : claim();
    for (bool run = true; run;) {
        if (!route_posted && idx >= a.n_logit) {
            // past this CTA's logit items: the consumers route next (an empty stage)
            uint32_t slot;
            if (!acquire(slot))
                break;
            s.tag[slot] = make_int2(TAG_ROUTE, 0);
            mbar_arrive(&s.full[slot]);
            ++st;
            route_posted = true;
            // the shared expert towards L2 only now: the router rows of the logit items,
            // on the routing critical path, go first
            if (a.has_shared)
                prefetch_shared(a);
        }
        if (!have_table && idx >= pre) {
            // the consumers' routing table (slots, pairs, counters) in shared memory
            if (!mbar_wait(s.tbar, 0)) {
                set_abort(a, s);
                break;
            }
            have_table = true;
            n_gu = a.n_logit + s.ctab->n_items_gateup;
            total = n_gu + s.ctab->n_items_down;
        }
        if (idx >= total) {
            uint32_t slot;
            if (acquire(slot)) {
                s.tag[slot] = make_int2(TAG_END, 0);  // end of work
                mbar_arrive(&s.full[slot]);
                ++st;
            }
            break;
        }
        int next = ahead;
        if (next >= 0)
            ahead = claim();  // used two items from now
        const DecItem it = work_item(a, s.stab, n_gu, idx);
        if (it.mode == MODE_LOGIT) {
            // chunk c: the item's token rows of x and its router rows over columns
            // [c * kc, c * kc + kcl)
            for (int c = 0; c < a.lg_nck; ++c) {
                uint32_t slot;
                if (!acquire(slot)) {
                    run = false;
                    break;
                }
                s.tag[slot] = make_int2(idx, c);
                s.sitem[slot] = it;
                {
                    const LogitItem li = logit_item(a, idx);
                    const int kc = a.lg_kc, k0 = c * kc, kcl = min(kc, a.d - k0);
                    const uint32_t rb = 4u * (uint32_t)kcl;
                    unsigned char *dst = s.ring + (size_t)slot * STAGE_BYTES;
                    mbar_arrive_expect_tx(&s.full[slot], (uint32_t)(li.ntok + li.ne) * rb);
                    for (int t = 0; t < li.ntok; ++t)
                        bulk_g2s(dst + (size_t)t * kc * 4, a.x + (long)(li.t0 + t) * a.d + k0, rb, &s.full[slot]);
                    for (int i = 0; i < li.ne; ++i)
                        bulk_g2s_hint(dst + (size_t)(a.lg_tb + i) * kc * 4, a.Wr + (long)(li.e0 + i) * a.d + k0, rb,
                                      &s.full[slot], pol);
                }
                ++st;
            }
            if (run && next < 0) {
                // the item's last stage has landed: claim the next item (and one ahead of
                // it unless it is a logit item too)
                if (!mbar_wait(&s.full[(st - 1) % NS], ((st - 1) / NS) & 1)) {
                    set_abort(a, s);
                    break;
                }
                next = claim();
                ahead = next < a.n_logit ? -1 : claim();
            }
            idx = next;
            continue;
        }
        const bool gu = it.mode == MODE_GATEUP;
        const colibri_expert ex = it.is_shared ? a.shared : s.stab[it.slot].ex;
        const int ng = it.kdim / G, spi = (ng + SG - 1) / SG;
        const int nq = spi * ((it.count + TCH - 1) / TCH);
        // the two row blocks: W1 and W3 at rb (gate/up), or W2 at rb and rb + 1 (down; the
        // second absent past the last row block)
        const unsigned char *wa, *wb;
        const float *sa_, *sb_;
        bool two = true;
        const int nsg = ng >> gsh;  // scale tiles a row block
        if (gu) {
            wa = ex.w1 + (size_t)it.rb * ng * 512;
            wb = ex.w3 + (size_t)it.rb * ng * 512;
            sa_ = ex.s1 + (size_t)it.rb * nsg * 32;
            sb_ = ex.s3 + (size_t)it.rb * nsg * 32;
        } else {
            two = it.rb + 1 < a.d / G;
            wa = ex.w2 + (size_t)it.rb * ng * 512;
            wb = wa + (size_t)ng * 512;
            sa_ = ex.s2 + (size_t)it.rb * nsg * 32;
            sb_ = sa_ + (size_t)nsg * 32;
        }
        for (int q = 0, ch = 0, k = 0; q < nq && run; ++q) {
            int flag = 0;
            if (!gu && k == 0 && (it.slot != hslot || ch != hch)) {
                // the chunk's rows of q8(h) into the next h buffer, once all rows of h of
                // its slot are published
                const int b = hsw % NH;
                if (hsw >= (uint32_t)NH && !mbar_wait(&s.hempty[b], ((hsw / NH) - 1) & 1)) {
                    set_abort(a, s);
                    run = false;
                    break;
                }
                if (!(it.slot < 64 && ((h_ready >> it.slot) & 1))) {
                    const int need = (it.is_shared ? a.shared_ffn : a.ffn) / G * it.count;
                    if (!wait_count_geq(a.done_gu + it.slot, need)) {
                        set_abort(a, s);
                        run = false;
                        break;
                    }
                    if (it.slot < 64)
                        h_ready |= 1ull << it.slot;
                }
                fence_proxy_async_global();  // h was written through the generic proxy
                const int nt = min(TCH, it.count - ch * TCH);
                unsigned char *hb = s.hbuf + (size_t)b * s.hb;
                int8_t *hcodes = reinterpret_cast<int8_t *>(hb);
                float *hsc = reinterpret_cast<float *>(hb + (size_t)TCH * a.fmax);
                int *hcr = reinterpret_cast<int *>(hsc + (size_t)TCH * a.hgs);
                mbar_arrive_expect_tx(&s.hfull[b], (uint32_t)(nt * (it.kdim + 8 * a.hgs)));
                for (int t = 0; t < nt; ++t) {
                    const long p = item_row(a, s, it, ch * TCH + t);
                    bulk_g2s(hcodes + (size_t)t * a.fmax, a.hq_eo + p * a.fmax, (uint32_t)it.kdim, &s.hfull[b]);
                    bulk_g2s(hsc + (size_t)t * a.hgs, a.hs + p * a.hgs, (uint32_t)(4 * a.hgs), &s.hfull[b]);
                    bulk_g2s(hcr + (size_t)t * a.hgs, a.hc + p * a.hgs, (uint32_t)(4 * a.hgs), &s.hfull[b]);
                }
                ++hsw;
                hslot = it.slot;
                hch = ch;
                flag = TAG_NEW_H;
            }
            uint32_t slot;
            if (!acquire(slot)) {
                run = false;
                break;
            }
            const int g0 = k * SG, n = min(SG, ng - g0);
            unsigned char *dst = s.ring + (size_t)slot * STAGE_BYTES;
            s.tag[slot] = make_int2(idx, k | (ch << 8) | flag);
            s.sitem[slot] = it;
            const int ns = n >> gsh, s0 = g0 >> gsh;  // the stage's scale tiles
            mbar_arrive_expect_tx(&s.full[slot], (uint32_t)((two ? 2 : 1) * (n * 512 + ns * 128)));
            bulk_g2s_hint(dst, wa + (size_t)g0 * 512, n * 512, &s.full[slot], pol);
            bulk_g2s_hint(dst + 2 * SG * 512, sa_ + (size_t)s0 * 32, ns * 128, &s.full[slot], pol);
            if (two) {
                bulk_g2s_hint(dst + SG * 512, wb + (size_t)g0 * 512, n * 512, &s.full[slot], pol);
                bulk_g2s_hint(dst + 2 * SG * 512 + SG * 128, sb_ + (size_t)s0 * 32, ns * 128, &s.full[slot], pol);
            }
            ++st;
            if (++k == spi) {
                k = 0;
                ++ch;
            }
        }
        idx = next;
    }
    // bounded waits for the copies issued, before the CTA exits
    const uint32_t n = st < (uint32_t)NS ? st : (uint32_t)NS;
    for (uint32_t k = 1; k <= n; ++k) {
        const uint32_t q = st - k;
        mbar_wait(&s.full[q % NS], (q / NS) & 1);
    }
    if (hsw > 0)
        mbar_wait(&s.hfull[(hsw - 1) % NH], ((hsw - 1) / NH) & 1);
}

// ---------------- epilogue warp e: the chunks that used partial-sum buffer e ----------------
// The epilogue warps' first job, while the consumers stream the logit items: this CTA's
// share of the q8 of x (one warp per group of 32 or 64 elements, lane k holding element k
// and k + 32, groups blockIdx.x * NE_MAX + e, ...), written to the workspace as plain
// codes and scales and as the codes in even/odd word order with their corrections
// 8 * sum(codes) per 32 elements; each group is counted with the logit tasks on the
// routing counter.
__device__ void quantise_x(const DecodeArgs &a, int e, int lane)
{
    const int gq = a.group, halves = gq / G, gx = a.d / gq;
    const long n = (long)a.T * gx;
    int done = 0;
    for (long gw = (long)blockIdx.x * NE_MAX + e; gw < n; gw += (long)gridDim.x * NE_MAX) {
        const long t = gw / gx, g = gw - t * gx;
        const long base = t * a.d + g * gq;
        float x[2];
        float m = 0.0f;
        for (int h = 0; h < halves; ++h) {
            x[h] = __ldcg(a.x + base + h * G + lane);  // in a layer stack, written in this launch
            m = fmaxf(m, fabsf(x[h]));
        }
        const float amax = warp_max(m);
        const float dd = __fdiv_rn(amax, 127.0f), rd = __frcp_rn(dd);
        for (int h = 0; h < halves; ++h) {
            const int q = q8_code_r(x[h], dd, rd);
            a.qx[base + h * G + lane] = (int8_t)q;
            a.xq_eo[base + h * G + eo_pos(lane)] = (int8_t)q;
            const int sq = warp_sum_i(q);
            if (lane == 0)
                a.xc[t * (a.d / G) + g * halves + h] = 8 * sq;
        }
        if (lane == 0)
            a.sx[gw] = dd;
        ++done;
    }
    if (done) {
        __threadfence();
        __syncwarp();
        if (lane == 0)
            atomicAdd(a.route_done, done);
    }
}

template <int TCH>
__device__ void run_epilogue(const DecodeArgs &a, const RingSmem &s, int e, int lane)
{
    constexpr int PART = NC * 2 * TCH * 32;
    const float *pb = s.part + (size_t)e * PART;
    for (uint32_t k = 0;; ++k) {
        if (!mbar_wait(&s.pfull[e], k & 1)) {
            if (lane == 0)
                set_abort(a, s);
            return;
        }
        const ChunkDesc *dp = s.desc + e;
        const int mode = dp->mode;
        if (mode < 0)
            return;  // end of work
        const int slot = dp->slot, rb = dp->rb, nt = dp->nt;
        int published = 0;  // rows of h (32-row blocks x tokens) whose q8 this chunk completed
        for (int t = 0; t < nt; ++t) {
            const long r = dp->orow[t];
            if (mode == MODE_GATEUP) {
                float gt = 0.0f, up = 0.0f;
                for (int w = 0; w < NC; ++w) {
                    gt += pb[((w * 2 + 0) * TCH + t) * 32 + lane];
                    up += pb[((w * 2 + 1) * TCH + t) * 32 + lane];
                }
                const float h = gt / (1.0f + expf(-gt)) * up;
                if (a.group == 64) {
                    // the 64-group of h spans row blocks rb & ~1 and rb | 1: the item that
                    // finishes second quantises both halves
                    a.hf[r * a.fmax + (long)rb * G + lane] = h;
                    __threadfence();
                    __syncwarp();
                    int second = 0;
                    if (lane == 0)
                        second = atomicAdd(a.hpair + r * (a.fmax / 64) + (rb >> 1), 1) == 1;
                    if (__shfl_sync(FULL, second, 0)) {
                        __threadfence();
                        const float hp = __ldcg(a.hf + r * a.fmax + (long)(rb ^ 1) * G + lane);
                        const float h0 = (rb & 1) ? hp : h, h1 = (rb & 1) ? h : hp;
                        const float amax = warp_max(fmaxf(fabsf(h0), fabsf(h1)));
                        const float dd = __fdiv_rn(amax, 127.0f), rd = __frcp_rn(dd);
                        const int q0 = q8_code_r(h0, dd, rd), q1 = q8_code_r(h1, dd, rd);
                        const long hb = r * a.fmax + (long)(rb >> 1) * 64;
                        a.hq[hb + lane] = (int8_t)q0;
                        a.hq[hb + G + lane] = (int8_t)q1;
                        a.hq_eo[hb + eo_pos(lane)] = (int8_t)q0;
                        a.hq_eo[hb + G + eo_pos(lane)] = (int8_t)q1;
                        const int s0 = warp_sum_i(q0), s1 = warp_sum_i(q1);
                        if (lane == 0) {
                            a.hs[r * a.hgs + (rb >> 1)] = dd;
                            a.hc[r * a.hgs + (rb & ~1)] = 8 * s0;
                            a.hc[r * a.hgs + (rb | 1)] = 8 * s1;
                        }
                        published += 2;
                    }
                } else {
                    const float amax = warp_max(fabsf(h));
                    const float dd = __fdiv_rn(amax, 127.0f);
                    const int q = q8_code_r(h, dd, __frcp_rn(dd));
                    const long hb = r * a.fmax + (long)rb * G;
                    a.hq[hb + lane] = (int8_t)q;
                    a.hq_eo[hb + eo_pos(lane)] = (int8_t)q;
                    const int sq = warp_sum_i(q);
                    if (lane == 0) {
                        a.hs[r * a.hgs + rb] = dd;
                        a.hc[r * a.hgs + rb] = 8 * sq;
                    }
                    published += 1;
                }
            } else {
                float y0 = 0.0f, y1 = 0.0f;
                for (int w = 0; w < NC; ++w) {
                    y0 += pb[((w * 2 + 0) * TCH + t) * 32 + lane];
                    y1 += pb[((w * 2 + 1) * TCH + t) * 32 + lane];
                }
                a.y[r * a.d + (long)rb * G + lane] = y0;
                if (rb + 1 < a.d / G)
                    a.y[r * a.d + (long)(rb + 1) * G + lane] = y1;
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&s.pempty[e]);  // the consumers may refill the buffer
        __threadfence();                // this chunk's rows are visible device-wide
        __syncwarp();
        if (mode == MODE_GATEUP) {
            if (lane == 0 && published)
                atomicAdd(a.done_gu + slot, published);
            continue;
        }
        // each of the item's row blocks of d: the epilogue that completes it combines it
        for (int b = rb; b < rb + 2 && b < a.d / G; ++b) {
            int last = 0;
            if (lane == 0) {
                last = atomicAdd(a.done_rb + b, nt) + nt == s.ctab->n_rows;
                if (last)
                    __threadfence();
            }
            if (__shfl_sync(FULL, last, 0)) {
                const long col = (long)b * G + lane;
                for (int t = 0; t < a.T; ++t) {
                    float o = a.has_shared ? __ldcg(a.y + ((long)a.T * a.K + t) * a.d + col) : 0.0f;
                    for (int i = 0; i < a.K; ++i)
                        o = fmaf(s.wtab[t * a.K + i], __ldcg(a.y + ((long)t * a.K + i) * a.d + col), o);
                    a.out[(long)t * a.d + col] = o;
                }
            }
        }
    }
}

// ---------------- consumer warps ----------------
template <int TCH>
__device__ void run_consumers(const DecodeArgs &a, const RingSmem &s, int warp, int lane)
{
    const int NBUF = a.nbuf;
    constexpr int PART = NC * 2 * TCH * 32;
    const int NS = a.ring, NH = a.nh;
    const int tid = threadIdx.x;
    uint32_t cph = 0;  // consumer barrier phase
    grid_dep_wait();   // the activations are in
    int8_t *xcodes = reinterpret_cast<int8_t *>(s.act);
    float *xsc = reinterpret_cast<float *>(s.act + x_sc_off(a.d, TCH));
    int *xcr = reinterpret_cast<int *>(s.act + x_cr_off(a.d, TCH));
    // q8 of x: all T tokens in the staging area when one chunk holds them, quantised by the
    // epilogue warps at the start (xbar; waited for at the routing stage), else each
    // chunk's tokens when it starts
    const bool x_all = a.T <= TCH;
    int xrows[TCH];  // token of each staged x row
#pragma unroll
    for (int t = 0; t < TCH; ++t)
        xrows[t] = x_all && t < a.T ? t : -1;
    bool x_staged = x_all;
    uint32_t chunk = 0;  // chunks handed to the epilogue (buffer chunk % NBUF)
    uint32_t hsw = 0;    // h buffers entered
    int cur_h = 0;
    int cur = -1, spi = 1, ng = 1;
    DecItem it{};
    int rows[TCH];
    int orow = -1;  // lane t < nt: pair row of the chunk's t-th token
    float acc[2][TCH];
    float *lacc = s.part + (size_t)warp * LT * 32;  // this warp's logit chains
    const int gsh = a.group == 64 ? 1 : 0;          // 32-column tile -> group
    // a buffer's previous chunk must have been read before it is written again
    const int nb_shift = NBUF == 4 ? 2 : 1;  // NBUF is 2 or 4
    auto buffer_free = [&](int b) -> bool {
        if (chunk >= (uint32_t)NBUF && !mbar_wait(&s.pempty[b], ((chunk >> nb_shift) - 1) & 1)) {
            if (lane == 0)
                set_abort(a, s);
            return false;
        }
        return true;
    };
    // the ring position of the next stage, kept incrementally (no division on this path)
    int nslot = 0;
    uint32_t nphase = 0;
    for (;;) {
        const int slot = nslot;
        const uint32_t phase = nphase;
        if (++nslot == NS) {
            nslot = 0;
            nphase ^= 1u;
        }
        if (!mbar_wait(&s.full[slot], phase)) {
            if (lane == 0)
                set_abort(a, s);
            return;
        }
        const int2 tag = s.tag[slot];
        if (tag.x == TAG_ROUTE) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s.empty[slot]);
            if (!route_cta(a, s, cph, tid, warp, lane))
                return;
            continue;
        }
        if (tag.x < 0) {
            // end of work: one end descriptor into every buffer, in buffer order
            for (int j = 0; j < NBUF; ++j, ++chunk) {
                const int b = chunk & (NBUF - 1);
                if (!buffer_free(b))
                    return;
                if (tid == 0)
                    s.desc[b].mode = -1;
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s.pfull[b]);
            }
            return;
        }
        if (tag.x != cur) {
            cur = tag.x;
            it = s.sitem[slot];  // decoded once, by the producer
            ng = it.kdim / G;
            spi = (ng + SG - 1) / SG;
        }
        const unsigned char *stg = s.ring + (size_t)slot * STAGE_BYTES;
        if (it.mode == MODE_LOGIT) {
            const int c = tag.y;
            logit_chunk(stg, a, cur, c, lacc, warp, lane);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s.empty[slot]);
            if (c != a.lg_nck - 1)
                continue;
            // end of the item: write its scores and count its tasks (the routing stages of
            // all CTAs wait for every task of the layer)
            const int nw = logit_finish(a, cur, lacc, warp, lane);
            __threadfence();
            __syncwarp();
            if (lane == 0 && nw > 0)
                atomicAdd(a.route_done, nw);
            continue;
        }
        const int k = tag.y & 255, ch = (tag.y >> 8) & 255;  // stage in the chunk, chunk
        const int c0 = ch * TCH, nt = min(TCH, it.count - c0);
        if (k == 0) {
            orow = lane < nt ? item_row(a, s, it, c0 + lane) : -1;
            if (it.mode == MODE_GATEUP) {
                int tok[TCH];
#pragma unroll
                for (int t = 0; t < TCH; ++t) {
                    const int p = __shfl_sync(FULL, orow, t);
                    tok[t] = t < nt ? (it.is_shared ? c0 + t : p / a.K) : -1;
                }
                bool same = x_staged;
                if (!x_all) {
#pragma unroll
                    for (int t = 0; t < TCH; ++t)
                        same &= xrows[t] == tok[t];
                }
                if (!same) {
                    // q8 of this chunk's tokens into the staging area, every warp alike
                    if (!consumers_sync(s, cph, lane))
                        return;
#pragma unroll
                    for (int t = 0; t < TCH; ++t)
                        xrows[t] = tok[t];
                    stage_x_rows<TCH>(a, xcodes, xsc, xcr, xrows, nt, tid);
                    if (!consumers_sync(s, cph, lane))
                        return;
                    x_staged = true;
                }
#pragma unroll
                for (int t = 0; t < TCH; ++t)
                    rows[t] = x_all ? (tok[t] < 0 ? 0 : tok[t]) : t;
            } else {
                if (tag.y & TAG_NEW_H) {
                    // leave the previous h buffer, enter the next one
                    __syncwarp();
                    if (hsw > 0 && lane == 0)
                        mbar_arrive(&s.hempty[(hsw - 1) % NH]);
                    if (!mbar_wait(&s.hfull[hsw % NH], (hsw / NH) & 1)) {
                        if (lane == 0)
                            set_abort(a, s);
                        return;
                    }
                    cur_h = hsw % NH;
                    ++hsw;
                }
#pragma unroll
                for (int t = 0; t < TCH; ++t)
                    rows[t] = t;
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int t = 0; t < TCH; ++t)
                    acc[m][t] = 0.0f;
        }
        if (it.mode == MODE_GATEUP) {
            consume<TCH>(stg, xcodes, xsc, xcr, a.d, a.d / G, a.d / a.group, gsh, rows, ng, k * SG, nt, warp, lane,
                         acc);
        } else {
            const unsigned char *hb = s.hbuf + (size_t)cur_h * s.hb;
            const int8_t *hcodes = reinterpret_cast<const int8_t *>(hb);
            const float *hsc = reinterpret_cast<const float *>(hb + (size_t)TCH * a.fmax);
            const int *hcr = reinterpret_cast<const int *>(hsc + (size_t)TCH * a.hgs);
            consume<TCH>(stg, hcodes, hsc, hcr, a.fmax, a.hgs, a.hgs, gsh, rows, ng, k * SG, nt, warp, lane, acc);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&s.empty[slot]);
        if (k != spi - 1)
            continue;

        // ---- end of a chunk: hand the partial sums to the epilogue warp of the buffer ----
        const int b = chunk & (NBUF - 1);
        if (!buffer_free(b))
            return;
        float *pb = s.part + (size_t)b * PART;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int t = 0; t < TCH; ++t)
                if (t < nt)
                    pb[((warp * 2 + m) * TCH + t) * 32 + lane] = acc[m][t];
        if (warp == 0) {
            ChunkDesc *dp = s.desc + b;
            if (lane < nt)
                dp->orow[lane] = orow;
            if (lane == 0) {
                dp->mode = it.mode;
                dp->slot = it.slot;
                dp->rb = it.rb;
                dp->nt = nt;
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&s.pfull[b]);
        ++chunk;
    }
}

}  // namespace

// The CTA's mbarriers for one layer (thread 0); `again` ends the previous layer's first.
__device__ void init_barriers(const DecodeArgs &a, const RingSmem &s, bool again)
{
    auto init = [&](uint64_t *b, uint32_t count) {
        if (again)
            mbar_inval(b);
        mbar_init(b, count);
    };
    for (int i = 0; i < a.ring; ++i) {
        init(&s.full[i], 1);
        init(&s.empty[i], NC);
    }
    for (int i = 0; i < a.nh; ++i) {
        init(&s.hfull[i], 1);
        init(&s.hempty[i], NC);
    }
    init(s.cbar, NC);
    init(s.tbar, 1);
    init(s.xbar, 1);
    for (int i = 0; i < a.nbuf; ++i) {
        init(&s.pfull[i], NC);
        init(&s.pempty[i], 1);
    }
    s.flags[0] = 0;
    fence_mbar_init();
}

// One layer on this CTA: the three roles.
template <int TCH>
__device__ __forceinline__ void run_layer(const DecodeArgs &a, const RingSmem &s, int warp, int lane)
{
    if (warp == NC) {
        if (lane == 0)
            run_producer<TCH>(a, s);
    } else if (warp > NC) {
        grid_dep_wait();  // the activations are in
        quantise_x(a, warp - NC - 1, lane);
        if (warp - NC - 1 < a.nbuf)
            run_epilogue<TCH>(a, s, warp - NC - 1, lane);
    } else {
        run_consumers<TCH>(a, s, warp, lane);
    }
}

template <int TCH>
__global__ void __launch_bounds__((NC + 1 + NE_MAX) * 32, 1) k_decode(DecodeArgs a)
{
    static_assert(TCH <= 8, "chunk descriptors hold 8 rows");  // launched with 1, 2 or 4
    extern __shared__ __align__(128) unsigned char sm[];
    const RingSmem s = carve(sm, a, TCH);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0)
        init_barriers(a, s, false);
    __syncthreads();
    run_layer<TCH>(a, s, warp, lane);
}

// This CTA's share of the next layer's router matrix and shared expert, sent towards L2
// while the current layer drains.
__device__ void prefetch_next_layer(const DecodeArgs &n)
{
    if (n.has_shared)
        prefetch_shared(n);
    if (n.Wr && !n.ids_given) {
        const size_t bytes = 4 * (size_t)n.E * n.d;
        const size_t share = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
        const size_t b0 = share * blockIdx.x;
        if (b0 < bytes)
            prefetch_l2(reinterpret_cast<const char *>(n.Wr) + b0, (uint32_t)min(share, bytes - b0));
    }
}

// Layers 0..L-1 in one launch. Between layers every CTA arrives on a grid barrier (a
// device counter, bounded wait): layer l + 1 starts only when layer l's output, its
// activations, is complete everywhere. Layer l uses control-word area l % 2; CTA 0 clears
// the other area at the start of layer l >= 1 for layer l + 1 (the launch's memset cleared
// both for layers 0 and 1). A CTA that gave up on a wait still arrives; after the
// barrier every CTA stops if the error word is set.
template <int TCH>
__global__ void __launch_bounds__((NC + 1 + NE_MAX) * 32, 1) k_decode_stack(const __grid_constant__ DecodeStack p)
{
    extern __shared__ __align__(128) unsigned char sm[];
    const RingSmem s = carve(sm, p.layer[0], TCH);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int l = 0; l < p.L; ++l) {
        const DecodeArgs &a = p.layer[l];
        if (blockIdx.x == 0 && l >= 1 && l + 1 < p.L) {
            int *z = p.sync_area[(l + 1) & 1];
            for (int i = threadIdx.x; i < p.sync_words; i += blockDim.x)
                z[i] = 0;
        }
        if (threadIdx.x == 0)
            init_barriers(a, s, l > 0);
        if (l > 0 && warp == NC && lane == 0)
            fence_proxy_async_global();  // the previous layer's output is read by bulk copies
        __syncthreads();
        run_layer<TCH>(a, s, warp, lane);
        if (l + 1 == p.L)
            break;
        if (warp == NC && lane == 0)
            prefetch_next_layer(p.layer[l + 1]);
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(p.bar, 1);
            const bool ok = wait_count_geq(p.bar, (int)gridDim.x * (l + 1));
            if (!ok)
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
            __threadfence();
            s.flags[1] = ok && ld_acquire_gpu(a.err) == 0;
        }
        __syncthreads();
        if (!s.flags[1])
            break;
    }
}

// ---- host-side dispatch -----------------------------------------------------------

namespace {

// Ring stages (and h and partial-sum buffers) for chunks of TCH tokens; 0 if fewer than
// two 40 KB stages fit.
template <int TCH>
int ring_for(DecodeArgs &a)
{
    // partial-sum buffers (= epilogue warps): 4 for chunks of at most 2 tokens, else 2;
    // then the most ring stages beside the rest, with 3 h buffers if that still leaves 4
    // stages, else 2 (measured: more buffers beat a fifth stage)
    const int nb = TCH <= 2 ? 4 : 2;
    int best_ns = 0, best_nh = 2;
    for (int nh = NH_MAX; nh >= 2; --nh) {
        int ns = MAX_RING;
        while (ns >= 2 && ring_layout(a, ns, nh, nb, TCH).total > SMEM_BUDGET)
            --ns;
        if (ns > best_ns) {
            best_ns = ns;
            best_nh = nh;
        }
        if (ns >= 4)
            break;
    }
    if (best_ns < 2)
        return 0;
    a.ring = best_ns;
    a.nh = best_nh;
    a.nbuf = nb;
    a.tch = TCH;
    return best_ns;
}

// The SM count of the current device (cached per device, under a lock).
cudaError_t sm_count_of_current(int &n_sm)
{
    constexpr int MAX_DEV = 64;
    static std::mutex mu;
    static int sm_count[MAX_DEV] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= MAX_DEV)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (sm_count[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        sm_count[dev] = n;
    }
    n_sm = sm_count[dev];
    return cudaSuccess;
}

// Raises kernel fn's dynamic shared memory limit to `smem` if needed. Per device and
// kernel (slot), the largest size set so far is kept (the attribute belongs to the
// device's context), so that a call costs no query; host threads that launch at the same
// time take the lock, so the attribute and its record agree.
template <typename F>
cudaError_t ensure_smem(F fn, int slot, size_t smem)
{
    constexpr int MAX_DEV = 64, SLOTS = 8;
    static std::mutex mu;
    static size_t smem_set[MAX_DEV][SLOTS] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= MAX_DEV || slot < 0 || slot >= SLOTS)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (smem > smem_set[dev][slot]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        smem_set[dev][slot] = smem;
    }
    return cudaSuccess;
}

template <int TCH>
cudaError_t launch_stack_tch(const DecodeStack &p, int n_sm, cudaStream_t s)
{
    auto fn = k_decode_stack<TCH>;
    const DecodeArgs &a = p.layer[0];
    const size_t smem = ring_layout(a, a.ring, a.nh, a.nbuf, TCH).total;
    cudaError_t e = ensure_smem(fn, 4 + TCH / 2, smem);
    if (e != cudaSuccess)
        return e;
    // a cooperative launch: the grid barrier between layers needs every CTA resident
    // (one per SM), which the launch then guarantees or refuses
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_sm);
    cfg.blockDim = dim3((NC + 1 + NE_MAX) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e != cudaSuccess) {
        // a stream that cannot take a programmatic dependency: plain stream order
        (void)cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, fn, p);
    }
    return e;
}

template <int TCH>
cudaError_t launch_tch(DecodeArgs a, int n_sm, cudaStream_t s)
{
    auto fn = k_decode<TCH>;
    const size_t smem = ring_layout(a, a.ring, a.nh, a.nbuf, TCH).total;
    cudaError_t e = ensure_smem(fn, TCH / 2, smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_sm);
    cfg.blockDim = dim3((NC + 1 + NE_MAX) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, a);
    if (e != cudaSuccess) {
        // a stream that cannot take a programmatic dependency: plain stream order
        (void)cudaGetLastError();
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, fn, a);
    }
    return e;
}

// The logit items: ne router rows against tb tokens, streamed in K-chunks of kc columns
// ((tb + ne) rows of kc floats fill at most one stage). The choice minimises the rows a
// CTA streams before routing can start, (tb + ne) times the items per CTA, with at most
// LT tasks (expert, token) per consumer warp; ties go to fewer items.
void logit_geometry(DecodeArgs &a, int n_sm)
{
    int best = 0x7fffffff, best_items = 0, bne = 1, btb = 1;
    for (int ne = 1; ne <= 8 && ne <= a.E; ++ne) {
        for (int tb = 1; tb <= a.T; ++tb) {
            if (ne * tb > NC * LT || 4 * (tb + ne) * 32 > STAGE_BYTES)
                continue;
            const int items = ((a.E + ne - 1) / ne) * ((a.T + tb - 1) / tb);
            const int cost = ((items + n_sm - 1) / n_sm) * (tb + ne);
            if (cost < best || (cost == best && items < best_items)) {
                best = cost;
                best_items = items;
                bne = ne;
                btb = tb;
            }
        }
    }
    int kc = STAGE_BYTES / (4 * (btb + bne)) / 32 * 32;
    kc = kc > a.d ? a.d : kc;
    const int nck = (a.d + kc - 1) / kc;
    a.lg_ne = bne;
    a.lg_tb = btb;
    a.lg_kc = round_up((a.d + nck - 1) / nck, 32);  // the same chunk count, balanced
    a.lg_nck = (a.d + a.lg_kc - 1) / a.lg_kc;
    a.n_logit = a.ids_given ? 0 : best_items;
    // warps that select at once: two score rows of E floats and 32 picks each in
    // SEL_SCRATCH bytes
    const int per = 8 * ((a.E + 3) & ~3) + 128;
    int sw = SEL_SCRATCH / per;
    sw = sw < 1 ? 1 : sw;
    sw = sw > NC ? NC : sw;
    a.sel_warps = sw > a.T ? a.T : sw;
}

}  // namespace

int decode_hgs(int fmax)
{
    return round_up(fmax / G, 4);
}

// The launch geometry of a decode call (logit items, tokens per chunk, ring); returns the
// tokens per chunk, or 0 if no ring fits.
int decode_geometry(DecodeArgs &a, int n_sm)
{
    a.hgs = decode_hgs(a.fmax);
    logit_geometry(a, n_sm);
    // tokens per chunk: up to 4 (a slot with more tokens streams its weights once per
    // chunk, but the smaller x, h and partial-sum areas leave room for a deeper ring);
    // fewer when a large shape leaves no room for three ring stages
    const int want = a.T <= 1 ? 1 : a.T <= 2 ? 2 : 4;
    DecodeArgs c4 = a, c2 = a, c1 = a;
    const int n4 = want >= 4 ? ring_for<4>(c4) : 0;
    const int n2 = want >= 2 ? ring_for<2>(c2) : 0;
    const int n1 = ring_for<1>(c1);
    if (n4 >= 3 || (n4 >= 2 && n2 < 3 && n1 < 3)) {
        a = c4;
        return 4;
    }
    if (n2 >= 3 || (n2 >= 2 && n1 < 3)) {
        a = c2;
        return 2;
    }
    if (n1 >= 2) {
        a = c1;
        return 1;
    }
    return 0;
}

cudaError_t launch_decode(DecodeArgs a, cudaStream_t s)
{
    if (a.T <= 0)
        return cudaSuccess;
    int n_sm = 0;
    cudaError_t e = sm_count_of_current(n_sm);
    if (e != cudaSuccess)
        return e;
    switch (decode_geometry(a, n_sm)) {
    case 4:
        return launch_tch<4>(a, n_sm, s);
    case 2:
        return launch_tch<2>(a, n_sm, s);
    case 1:
        return launch_tch<1>(a, n_sm, s);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_stack(DecodeStack &p, cudaStream_t s)
{
    if (p.L < 1 || p.L > STACK_MAX)
        return cudaErrorInvalidValue;
    if (p.layer[0].T <= 0)
        return cudaSuccess;
    int n_sm = 0;
    cudaError_t e = sm_count_of_current(n_sm);
    if (e != cudaSuccess)
        return e;
    DecodeArgs g = p.layer[0];
    const int tch = decode_geometry(g, n_sm);
    for (int l = 0; l < p.L; ++l) {
        DecodeArgs &a = p.layer[l];
        a.ring = g.ring;
        a.nh = g.nh;
        a.nbuf = g.nbuf;
        a.tch = g.tch;
        a.hgs = g.hgs;
        a.lg_ne = g.lg_ne;
        a.lg_tb = g.lg_tb;
        a.lg_kc = g.lg_kc;
        a.lg_nck = g.lg_nck;
        a.n_logit = g.n_logit;
        a.sel_warps = g.sel_warps;
    }
    switch (tch) {
    case 4:
        return launch_stack_tch<4>(p, n_sm, s);
    case 2:
        return launch_stack_tch<2>(p, n_sm, s);
    case 1:
        return launch_stack_tch<1>(p, n_sm, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace clb
