// Per-layer routing-control pass of the expert cache: one CTA per call.
//
// FreeToken explainer, section 10 "Dynamic Scheduling Without Giving Up CUDA
// Graphs", and deepmox chapter "The Expert Cache That Follows the Router",
// section "How residency follows demand without leaving the device": the
// pass deduplicates the routed experts, classifies each flat id layer*E+e as
// hit or miss through slot_for_id, derives the fill count q (explainer
// section 5, q* = m*B_P/B_H; txtmix: at least one fill), picks the fill set
// F and the LRU victims, updates the maps and recency, rewrites the route ids
// to slot ids and leaves fixed-size worklists with a valid count for the
// expert kernels -- all on the device, without a host round trip.
//
// Conventions of this implementation (the pages leave them open):
//   top-k by logit descending, lower id first on ties; gates = softmax over
//   the k selected logits (fp32); q0 = round((m*B_P)/B_H) in fp64, halves away
//   from zero; q = min(clamp(q0,1,m), S-h); fill order = routed-token count
//   descending, lower id first; a clock incremented per pass stamps hits and
//   fills; victims = the q smallest (stamp, slot) among slots not holding a
//   hit; the i-th fill expert takes the i-th victim.
//
// Latency design: every global read the pass needs (logits, the layer's row
// of slot_for_id, the stamps and owners of all slots, the clock) is issued at
// entry and lands in shared memory; the rest runs on shared memory.  Victim
// discovery works on (stamp, slot) keys after the hits' stamps were refreshed
// to the current clock -- every non-hit slot then has a smaller stamp than
// every hit slot, so the q smallest keys over all slots are exactly the q
// smallest non-hit keys (q <= S - h).  Small q: q block-wide arg-min rounds;
// larger q: one radix select over the stamps (the txtmix write-up's "one scan
// yields K LRU candidates") then a rank sort of the candidates.
#include "ft_common.cuh"

#include <math.h>

namespace {

constexpr int CTL_THREADS = 512;
constexpr int CTL_WARPS = CTL_THREADS / 32;
constexpr int SMALL_Q = 8;

struct CtlShared {
    int bad;
    int u, h, m;
    int q0, q1, q;
    unsigned clk;
    int sel_bin, sel_before;
    int ugpu, nassign;
    int carry0, carry1;
    int warp_tot[CTL_WARPS];
    unsigned long long warp_key[CTL_WARPS];
    int hist[256];
};

// Block-wide exclusive scan of one int per thread.
__device__ int block_excl_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = lane < CTL_WARPS ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < CTL_WARPS) warp_tot[lane] = w;
    }
    __syncthreads();
    const int base = wid ? warp_tot[wid - 1] : 0;
    const int tot = warp_tot[CTL_WARPS - 1];
    __syncthreads();
    *total = tot;
    return base + x - v;
}

// Order-preserving unsigned key of a finite float (larger value, larger
// key); -0 and +0 map to the same key.
__device__ __forceinline__ unsigned ordered_key(float v) {
    const unsigned u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
    return a < b ? a : b;
}

// Running totals of the context (read by the host between calls): reductions
// without a return value, so the pass does not wait on their loads.
__device__ __forceinline__ void add_counters(unsigned long long* c, int u, int h, int m, int q, int nassign) {
    atomicAdd(&c[CNT_CALLS], 1ull);
    atomicAdd(&c[CNT_UNIQUE], (unsigned long long)u);
    atomicAdd(&c[CNT_HITS], (unsigned long long)h);
    atomicAdd(&c[CNT_MISSES], (unsigned long long)m);
    atomicAdd(&c[CNT_FILLS], (unsigned long long)q);
    atomicAdd(&c[CNT_CPU], (unsigned long long)(m - q));
    atomicAdd(&c[CNT_ASSIGN], (unsigned long long)nassign);
}

// a4: q = min(clamp(q0, 1, m), S - h) with q0 = round(m * B_P / B_H) in fp64
// (halves away from zero); the host tabulates q0 for m <= E.
__device__ int fill_count(const CtlParams& p, int m, int h, int S, int& q0, int& q1) {
    q0 = q1 = 0;
    if (m <= 0) return 0;
    if (m < p.q0_n) {
        q0 = p.q0tab[m];  // the same fp64 expression, evaluated on the host per m
    } else {
        const double x = __ddiv_rn(__dmul_rn((double)m, p.B_P), p.B_H);
        const double r = round(x);  // halves away from zero
        q0 = r > 1.0e9 ? 1000000000 : (int)r;
    }
    q1 = min(max(q0, 1), m);
    return max(min(q1, S - h), 0);
}

// a6: victims = the q smallest (stamp, slot) keys, into s_vict[0..q) in
// ascending key order; called by every thread of the block.  Small q: q
// block-wide arg-min rounds; larger q: a radix select of the q-th stamp, then
// a rank sort of the candidates below it.  Each taken slot's staged stamp is
// set to clk (the hits were refreshed to clk before the call), so no slot is
// taken twice.
__device__ void select_victims(CtlShared& sh, unsigned* s_stamp, int* s_vict, int* s_cslot, unsigned* s_cst,
                               const int S, const int q, const unsigned clk) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (q > 0 && q <= SMALL_Q) {
        for (int r = 0; r < q; ++r) {
            unsigned long long best = ~0ull;
            for (int s = tid; s < S; s += CTL_THREADS)
                best = umin64(best, ((unsigned long long)s_stamp[s] << 32) | (unsigned)s);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = umin64(best, __shfl_xor_sync(0xffffffffu, best, o));
            if (lane == 0) sh.warp_key[wid] = best;
            __syncthreads();
            if (wid == 0) {
                unsigned long long b = lane < CTL_WARPS ? sh.warp_key[lane] : ~0ull;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) b = umin64(b, __shfl_xor_sync(0xffffffffu, b, o));
                if (lane == 0) {
                    const int v = (int)(b & 0xffffffffu);
                    s_vict[r] = v;
                    s_stamp[v] = clk;  // taken: never the minimum again
                }
            }
            __syncthreads();
        }
    } else if (q > SMALL_Q) {
        unsigned prefix = 0u, pmask = 0u;
        int need = q;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += CTL_THREADS) sh.hist[i] = 0;
            __syncthreads();
            for (int s = tid; s < S; s += CTL_THREADS) {
                const unsigned st = s_stamp[s];
                if ((st & pmask) == prefix) atomicAdd(&sh.hist[(st >> shift) & 255u], 1);
            }
            __syncthreads();
            if (wid == 0) {
                int c[8];
                int sum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    c[i] = sh.hist[lane * 8 + i];
                    sum += c[i];
                }
                int incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const int excl = incl - sum;
                const unsigned ball = __ballot_sync(0xffffffffu, excl < need && need <= incl);
                if (lane == __ffs(ball) - 1) {
                    int run = excl, b = lane * 8 + 7;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (run + c[i] >= need) {
                            b = lane * 8 + i;
                            break;
                        }
                        run += c[i];
                    }
                    sh.sel_bin = b;
                    sh.sel_before = run;
                }
            }
            __syncthreads();
            prefix |= (unsigned)sh.sel_bin << shift;
            pmask |= 255u << shift;
            need -= sh.sel_before;
        }
        const unsigned tau = prefix;
        const int c_lt = q - need;  // slots with stamp < tau are all victims; `need` of stamp == tau
        if (tid == 0) {
            sh.carry0 = 0;
            sh.carry1 = 0;
        }
        __syncthreads();
        for (int s0 = 0; s0 < S; s0 += CTL_THREADS) {
            const int s = s0 + tid;
            const unsigned st = s < S ? s_stamp[s] : 0xffffffffu;
            const int flt = (s < S && st < tau) ? 1 : 0;
            const int feq = (s < S && st == tau) ? 1 : 0;
            int tot;
            const int ex = block_excl_scan(flt | (feq << 16), sh.warp_tot, &tot);
            const int ex_lt = (ex & 0xffff) + sh.carry0;
            const int ex_eq = (ex >> 16) + sh.carry1;
            if (flt) {
                s_cslot[ex_lt] = s;
                s_cst[ex_lt] = st;
            }
            if (feq && ex_eq < need) s_vict[c_lt + ex_eq] = s;
            __syncthreads();
            if (tid == 0) {
                sh.carry0 += tot & 0xffff;
                sh.carry1 += tot >> 16;
            }
            __syncthreads();
        }
        for (int i = tid; i < c_lt; i += CTL_THREADS) {
            const unsigned si = s_cst[i];
            const int li = s_cslot[i];
            int r = 0;
            for (int j = 0; j < c_lt; ++j) {
                const unsigned sj = s_cst[j];
                r += (sj < si) || (sj == si && s_cslot[j] < li);
            }
            s_vict[r] = li;
        }
        __syncthreads();
    }

}

__global__ void __launch_bounds__(CTL_THREADS, 1) route_ctl_kernel(CtlParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ CtlShared sh;
    const int T = p.T, k = p.k, E = p.E, S = p.S, TK = T * k;
    const int TW = (T + 63) >> 6;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int fbase = p.layer * E;

    unsigned long long* s_tmask = reinterpret_cast<unsigned long long*>(smem_raw);  // [E*TW]
    unsigned* s_stamp = reinterpret_cast<unsigned*>(s_tmask + (size_t)E * TW);     // [S]
    int* s_owner = reinterpret_cast<int*>(s_stamp + S);                             // [S]
    int* s_ids = s_owner + S;                                                        // [TK]
    float* s_g = reinterpret_cast<float*>(s_ids + TK);                               // [TK]
    int* s_cnt = reinterpret_cast<int*>(s_g + TK);                                   // [E]
    int* s_row = s_cnt + E;     // [E] slot_for_id row of this layer (before the pass)
    int* s_cls = s_row + E;     // [E] 0 not routed, 1 hit, 2 fill, 3 CPU (miss)
    int* s_slot = s_cls + E;    // [E] slot of a GPU expert
    int* s_order = s_slot + E;  // [E] misses by fill rank
    int* s_eoff = s_order + E;  // [E] first assignment of GPU expert e
    int* s_vict = s_eoff + E;   // [E] victims by rank
    int* s_cslot = s_vict + E;  // [E] radix path: candidates with stamp < tau
    unsigned* s_cst = reinterpret_cast<unsigned*>(s_cslot + E);  // [E]

    if (tid == 0) {
        sh.bad = 0;
        sh.u = sh.h = sh.m = 0;
    }
    __syncthreads();
    // ---- issue every global read of the pass
    for (int s = tid; s < S; s += CTL_THREADS) {
        s_stamp[s] = p.stamps[s];
        s_owner[s] = p.id_for_slot[s];
    }
    for (int e = tid; e < E; e += CTL_THREADS) {
        s_row[e] = p.slot_for_id[fbase + e];
        s_cnt[e] = 0;
        s_cls[e] = 0;
        s_slot[e] = -1;
    }
    for (int i = tid; i < E * TW; i += CTL_THREADS) s_tmask[i] = 0ull;
    if (tid == 0) sh.clk = *p.clock;

    // ---- a1: routing (top-k + softmax gates), or the given top-k
    if (p.logits) {
        for (int t = wid; t < T; t += CTL_WARPS) {
            const float* row = p.logits + (size_t)t * E;
            constexpr int RV = 8;  // values per lane held in registers (E <= 256)
            float vals[RV];
            bool bad = false;
#pragma unroll
            for (int i = 0; i < RV; ++i) {
                const int e = lane + 32 * i;
                vals[i] = e < E ? row[e] : -INFINITY;
                if (e < E && !isfinite(vals[i])) bad = true;
            }
            bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the shuffle loop
            unsigned used = 0;
            float sel_v = 0.f;
            int sel_e = 0;
            for (int j = 0; j < k && !bad; ++j) {
                float bv = -INFINITY;
                int be = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < RV; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && !((used >> i) & 1u)) {
                        const float v = vals[i];
                        if (v > bv || (v == bv && e < be)) {
                            bv = v;
                            be = e;
                        }
                    }
                }
                for (int i = RV; lane + 32 * i < E; ++i) {
                    if ((used >> i) & 1u) continue;
                    const int e = lane + 32 * i;
                    const float v = row[e];
                    if (v > bv || (v == bv && e < be)) {
                        bv = v;
                        be = e;
                    }
                }
                // warp arg-max as two reductions: the largest value (as an
                // order-preserving key, -0 folded into +0 so that equal values
                // tie), then the lowest id among the lanes holding it
                const unsigned key = ordered_key(bv);
                const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
                be = (int)__reduce_min_sync(0xffffffffu, key == kmax ? (unsigned)be : 0xffffffffu);
                bv = __shfl_sync(0xffffffffu, bv, be & 31);
                if (be >= E) {
                    bad = true;
                    break;
                }
                if ((be & 31) == lane) used |= 1u << (be >> 5);
                if (lane == j) {
                    sel_v = bv;
                    sel_e = be;
                }
            }
            if (__any_sync(0xffffffffu, bad)) {
                if (lane == 0) sh.bad = 1;
                continue;
            }
            const float v0 = __shfl_sync(0xffffffffu, sel_v, 0);
            const float ex = lane < k ? expf(sel_v - v0) : 0.f;
            const float den = ft::warp_sum(ex);
            if (lane < k) {
                const float g = ex / den;
                s_ids[t * k + lane] = sel_e;
                s_g[t * k + lane] = g;
                p.out_ids[t * k + lane] = sel_e;
                p.out_gates[t * k + lane] = g;
            }
        }
        __syncthreads();
    } else {
        for (int a = tid; a < TK; a += CTL_THREADS) {
            const int e = p.topk_ids[a];
            const float g = p.topk_w[a];
            if (e < 0 || e >= E || !isfinite(g)) sh.bad = 1;
            s_ids[a] = e;
            s_g[a] = g;
            p.out_ids[a] = e;
            p.out_gates[a] = g;
        }
        __syncthreads();
        for (int a = tid; a < TK; a += CTL_THREADS) {
            const int t = a / k, j = a - t * k;
            for (int j2 = 0; j2 < j; ++j2)
                if (s_ids[t * k + j2] == s_ids[a]) sh.bad = 1;
        }
        __syncthreads();
    }
    if (sh.bad) {
        for (int a = tid; a < TK; a += CTL_THREADS) {
            p.out_pos[a] = -1;
            p.out_slots[a] = -1;
        }
        if (tid == 0) {
            atomicOr(p.err, FT_DEVERR_ARG);
            for (int i = 0; i < INFO_WORDS; ++i) p.info[i] = 0;
            p.info[INFO_LAYER] = p.layer;
            p.info[INFO_T] = T;
            p.info[INFO_CLOCK] = (int)sh.clk;
            p.wl_off[0] = 0;
        }
        return;
    }

    // ---- small batches (T*k <= 32): one warp carries the pass, lane a
    // holding assignment a = t*k + j, with votes and shuffles in place of
    // the block-wide phases of the general path below; every warp joins for
    // the victim search only.  Same decisions and outputs as that path.
    if (TK <= 32) {
        constexpr unsigned FULL = 0xffffffffu;
        const bool act = lane < TK;
        int e = 0, n_e = 0, r = 0, cls = 0, sl = -1, ldr = 0;
        unsigned peers = 0, hitm = 0, fillm = 0;
        int q = 0;
        unsigned clk = 0;
        if (wid == 0) {
            // a2: dedup -- the lanes of one expert, its routed-token count, the first as leader
            e = act ? s_ids[lane] : -1 - lane;  // idle lanes: keys no routed id matches
            peers = __match_any_sync(FULL, e);
            ldr = __ffs(peers) - 1;
            n_e = __popc(peers);
            const bool leader = act && ldr == lane;
            // a3: classify against the layer's residency row
            if (leader) {
                sl = s_row[e];
                cls = sl >= 0 ? 1 : 3;
            }
            hitm = __ballot_sync(FULL, cls == 1);
            const unsigned missm = __ballot_sync(FULL, cls == 3);
            const int u = __popc(__ballot_sync(FULL, leader)), h = __popc(hitm), m = __popc(missm);
            // a5 order: rank of each miss by (count desc, id asc)
            for (int i = 0; i < TK; ++i) {
                const int e2 = __shfl_sync(FULL, e, i), n2 = __shfl_sync(FULL, n_e, i);
                if ((missm >> i) & 1u) r += (n2 > n_e) || (n2 == n_e && e2 < e);
            }
            // a4: q; the clock advances once per pass
            clk = sh.clk + 1u;
            int qq = 0;
            __syncwarp();
            if (lane == 0) {
                int q0, q1;
                qq = fill_count(p, m, h, S, q0, q1);
                sh.q0 = q0;
                sh.q1 = q1;
                sh.q = qq;
                sh.u = u;
                sh.h = h;
                sh.m = m;
                sh.clk = clk;
            }
            q = __shfl_sync(FULL, qq, 0);
            // a5: F = the first q misses, C = the rest; a7 (part): hit stamps
            if (cls == 3) {
                if (r < q) {
                    cls = 2;
                    p.out_F[r] = e;
                    s_order[r] = e;
                } else {
                    p.out_C[r - q] = e;
                }
            }
            if (cls == 1) {
                s_stamp[sl] = clk;
                p.stamps[sl] = clk;
            }
            fillm = __ballot_sync(FULL, cls == 2);
        }
        __syncthreads();
        // ---- a6: victims (every warp)
        select_victims(sh, s_stamp, s_vict, s_cslot, s_cst, S, sh.q, sh.clk);
        if (wid != 0) return;
        // ---- a7: evict the victims' owners, install F, stamp the fills
        if (lane < q) {
            const int f = s_order[lane];
            const int v = s_vict[lane];
            const int o = s_owner[v];
            if (o >= 0) p.slot_for_id[o] = -1;
            const int fid = fbase + f;
            p.id_for_slot[v] = fid;
            p.slot_for_id[fid] = v;
            p.stamps[v] = clk;
            p.ready[lane] = 0u;
            p.fill_slot[lane] = v;
            p.fill_fid[lane] = fid;
            p.out_victims[lane] = v;
        }
        if (cls == 2) sl = s_vict[r];
        // ---- a7: worklist -- the hits in ascending expert id, then the
        // fills in fill order; offsets are the routed-token counts before
        int hidx = 0, hoff = 0, foff = 0;
        for (int i = 0; i < TK; ++i) {
            const int e2 = __shfl_sync(FULL, e, i), n2 = __shfl_sync(FULL, n_e, i), r2 = __shfl_sync(FULL, r, i);
            if (((hitm >> i) & 1u) && e2 < e) {
                ++hidx;
                hoff += n2;
            }
            if (((fillm >> i) & 1u) && r2 < r) foff += n2;
        }
        const int hasg = (int)__reduce_add_sync(FULL, cls == 1 ? (unsigned)n_e : 0u);
        const int fasg = (int)__reduce_add_sync(FULL, cls == 2 ? (unsigned)n_e : 0u);
        const int nh = __popc(hitm);
        int eo = 0;
        if (cls == 1 || cls == 2) {
            const int ent = cls == 1 ? hidx : nh + r;
            eo = cls == 1 ? hoff : hasg + foff;
            p.wl_slot[ent] = sl;
            p.wl_fid[ent] = fbase + e;
            p.wl_fill[ent] = cls == 1 ? -1 : r;
            p.wl_off[ent] = eo;
        }
        // every assignment: its expert's class, slot and offset from the
        // leader; its rank among the expert's tokens (ascending with the lane)
        const int c2 = __shfl_sync(FULL, cls, ldr), s2 = __shfl_sync(FULL, sl, ldr), o2 = __shfl_sync(FULL, eo, ldr);
        if (act) {
            if (c2 == 1 || c2 == 2) {
                const int pos = o2 + __popc(peers & ((1u << lane) - 1u));
                p.as_tok[pos] = lane / k;
                p.as_gate[pos] = s_g[lane];
                p.out_pos[lane] = pos;
                p.out_slots[lane] = s2;
            } else {
                p.out_pos[lane] = -1;
                p.out_slots[lane] = -1;
            }
        }
        if (lane == 0) {
            const int ugpu = nh + q, nassign = hasg + fasg;
            p.wl_off[ugpu] = nassign;
            *p.clock = clk;
            int* I = p.info;
            I[INFO_LAYER] = p.layer;
            I[INFO_T] = T;
            I[INFO_U] = sh.u;
            I[INFO_H] = sh.h;
            I[INFO_M] = sh.m;
            I[INFO_Q0] = sh.q0;
            I[INFO_Q1] = sh.q1;
            I[INFO_Q] = q;
            I[INFO_NC] = sh.m - q;
            I[INFO_UGPU] = ugpu;
            I[INFO_NASSIGN] = nassign;
            I[INFO_CLOCK] = (int)clk;
            I[INFO_VALID] = 1;
            add_counters(p.counters, sh.u, sh.h, sh.m, q, nassign);
        }
        return;
    }

    // ---- a2: dedup -- routed-token count n_e and token membership masks
    for (int a = tid; a < TK; a += CTL_THREADS) {
        const int e = s_ids[a];
        const int t = a / k;
        atomicAdd(&s_cnt[e], 1);
        atomicOr(&s_tmask[(size_t)e * TW + (t >> 6)], 1ull << (t & 63));
    }
    __syncthreads();

    // ---- a3: classify against the residency row of this layer
    for (int e = tid; e < E; e += CTL_THREADS) {
        if (s_cnt[e] > 0) {
            const int sl = s_row[e];
            atomicAdd(&sh.u, 1);
            if (sl >= 0) {
                s_cls[e] = 1;
                s_slot[e] = sl;
                atomicAdd(&sh.h, 1);
            } else {
                s_cls[e] = 3;
                atomicAdd(&sh.m, 1);
            }
        }
    }
    __syncthreads();

    // ---- a5 (order): fill rank of every miss = (count desc, id asc); a4: q.
    // One warp per miss counts the misses that precede it, 32 ids at a time.
    for (int e = wid; e < E; e += CTL_WARPS) {
        if (s_cls[e] != 3) continue;  // warp-uniform
        const int ne = s_cnt[e];
        int r = 0;
        for (int e2 = lane; e2 < E; e2 += 32) {
            if (s_cls[e2] == 3) {
                const int n2 = s_cnt[e2];
                r += (n2 > ne) || (n2 == ne && e2 < e);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        if (lane == 0) s_order[r] = e;
    }
    if (tid == 0) {
        int q0, q1;
        const int q = fill_count(p, sh.m, sh.h, S, q0, q1);
        sh.q0 = q0;
        sh.q1 = q1;
        sh.q = q;
        sh.clk = sh.clk + 1u;
    }
    __syncthreads();
    const int q = sh.q, m = sh.m;
    const unsigned clk = sh.clk;

    // ---- a5: F = first q misses, C = the rest; a7 (part): refresh hit stamps
    for (int r = tid; r < m; r += CTL_THREADS) {
        const int e = s_order[r];
        if (r < q) {
            s_cls[e] = 2;
            p.out_F[r] = e;
        } else {
            p.out_C[r - q] = e;
        }
    }
    for (int e = tid; e < E; e += CTL_THREADS) {
        if (s_cls[e] == 1) {
            s_stamp[s_slot[e]] = clk;
            p.stamps[s_slot[e]] = clk;
        }
    }
    __syncthreads();

    // ---- a6: victims = q smallest (stamp, slot)
    select_victims(sh, s_stamp, s_vict, s_cslot, s_cst, S, q, clk);

    // ---- a7: evict the victims' owners, install F, stamp the fills
    for (int i = tid; i < q; i += CTL_THREADS) {
        const int f = s_order[i];
        const int v = s_vict[i];
        const int o = s_owner[v];
        if (o >= 0) p.slot_for_id[o] = -1;
        const int fid = fbase + f;
        p.id_for_slot[v] = fid;
        p.slot_for_id[fid] = v;
        p.stamps[v] = clk;
        s_slot[f] = v;
        p.ready[i] = 0u;
        p.fill_slot[i] = v;
        p.fill_fid[i] = fid;
        p.out_victims[i] = v;
    }
    __syncthreads();

    // ---- a7: GPU worklist and the slot rewrite.  Entries: the hits in
    // ascending expert id, then the fills in fill order (the expert kernel
    // computes the hits while the fills are still landing).  One warp scans
    // the entry numbers and the assignment offsets, 32 experts at a time.
    if (wid == 0) {
        int nh = 0, off = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int hit = (e < E && s_cls[e] == 1) ? 1 : 0;
            const int cnt = hit ? s_cnt[e] : 0;
            int xh = hit, xc = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yh = __shfl_up_sync(0xffffffffu, xh, o);
                const int yc = __shfl_up_sync(0xffffffffu, xc, o);
                if (lane >= o) {
                    xh += yh;
                    xc += yc;
                }
            }
            if (hit) {
                const int ent = nh + xh - 1;
                const int eo = off + xc - cnt;
                s_eoff[e] = eo;
                p.wl_slot[ent] = s_slot[e];
                p.wl_fid[ent] = fbase + e;
                p.wl_fill[ent] = -1;
                p.wl_off[ent] = eo;
            }
            nh += __shfl_sync(0xffffffffu, xh, 31);
            off += __shfl_sync(0xffffffffu, xc, 31);
        }
        for (int i0 = 0; i0 < q; i0 += 32) {
            const int i = i0 + lane;
            const int e = i < q ? s_order[i] : -1;
            const int cnt = e >= 0 ? s_cnt[e] : 0;
            int xc = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yc = __shfl_up_sync(0xffffffffu, xc, o);
                if (lane >= o) xc += yc;
            }
            if (e >= 0) {
                const int ent = nh + i;
                const int eo = off + xc - cnt;
                s_eoff[e] = eo;
                p.wl_slot[ent] = s_slot[e];
                p.wl_fid[ent] = fbase + e;
                p.wl_fill[ent] = i;
                p.wl_off[ent] = eo;
            }
            off += __shfl_sync(0xffffffffu, xc, 31);
        }
        if (lane == 0) {
            sh.ugpu = nh + q;
            sh.nassign = off;
            p.wl_off[nh + q] = off;
            *p.clock = clk;
        }
    }
    __syncthreads();
    for (int a = tid; a < TK; a += CTL_THREADS) {
        const int e = s_ids[a];
        const int t = a / k;
        const int c = s_cls[e];
        if (c == 1 || c == 2) {
            const unsigned long long* mk = s_tmask + (size_t)e * TW;
            int rank = 0;
            for (int w = 0; w < (t >> 6); ++w) rank += __popcll(mk[w]);
            rank += __popcll(mk[t >> 6] & ((1ull << (t & 63)) - 1ull));
            const int pos = s_eoff[e] + rank;
            p.as_tok[pos] = t;
            p.as_gate[pos] = s_g[a];
            p.out_pos[a] = pos;
            p.out_slots[a] = s_slot[e];
        } else {
            p.out_pos[a] = -1;
            p.out_slots[a] = -1;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int* I = p.info;
        I[INFO_LAYER] = p.layer;
        I[INFO_T] = T;
        I[INFO_U] = sh.u;
        I[INFO_H] = sh.h;
        I[INFO_M] = sh.m;
        I[INFO_Q0] = sh.q0;
        I[INFO_Q1] = sh.q1;
        I[INFO_Q] = q;
        I[INFO_NC] = sh.m - q;
        I[INFO_UGPU] = sh.ugpu;
        I[INFO_NASSIGN] = sh.nassign;
        I[INFO_CLOCK] = (int)clk;
        I[INFO_VALID] = 1;
        add_counters(p.counters, sh.u, sh.h, sh.m, q, sh.nassign);
    }
}

}  // namespace

size_t route_ctl_smem_bytes(int T, int k, int E, int S) {
    const size_t TW = (T + 63) / 64;
    return (size_t)E * TW * 8 + (size_t)S * 8 + (size_t)T * k * 8 + (size_t)E * 13 * 4;
}

cudaError_t launch_route_ctl(const CtlParams& p, cudaStream_t s) {
    const size_t smem = route_ctl_smem_bytes(p.T, p.k, p.E, p.S);
    cudaError_t e = ensure_dynamic_smem((const void*)route_ctl_kernel, smem);
    if (e != cudaSuccess) return e;
    route_ctl_kernel<<<1, CTL_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}
