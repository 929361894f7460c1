// decode_cta.cuh -- one CTA's share of the decode attention over a block-paged KV cache
// (the body of paged_decode_kernel, also run by the decode CTAs of paged_varlen_kernel).
//
// Method ("vLLM推理引擎架构PagedAttention机制与高吞吐推理", lpnh.cn, §2.3 PagedAttention
// Kernel): for each sequence, find each token's KV block through block_tables, score
// the query against the keys inside the block, and accumulate across blocks.  The
// accumulation across blocks is an online softmax in fp32 (running max m, running sum
// l, rescaled output o); parts of one context computed by different thread blocks are
// merged with their log-sum-exp weights.
//
// GB300 design
//  * Work is the flat list of (sequence, KV-head tile, 16-token block) units.  A
//    persistent grid of one CTA per SM takes an equal contiguous share of it (+-1
//    block), so a 32k context and a 500-token one cost the same per block and no SM
//    idles in a tail.  A CTA's share can start or end inside a sequence: those parts go
//    to a workspace slot and the merge kernel combines them.
//  * A CTA covers all KV heads of its tile (8 for Llama-70B shapes), so each pool block
//    it touches is read as whole 16-token x 2 KiB rows: one producer warp streams K and
//    V of each block with TMA (128-byte swizzled, evict-first) into a ring of shared
//    memory stages guarded by mbarriers; the block id comes from the block table.
//  * One consumer warp per (KV head, up to 16 query heads): GQA puts the group's query
//    heads on the N of m16n8k16 tensor-core MMAs and the block's 16 tokens on M, so one
//    K/V read from shared memory serves the whole group with no padded rows (8 heads
//    fill N): S^T = K Q^T and O^T += V^T P^T (bf16t_block.cuh; fp8_block.cuh for an FP8
//    cache).
//  * No thread ever waits on another CTA.  Every mbarrier wait is bounded in time and
//    reports PKV_DEVERR_TIMEOUT instead of hanging.
#pragma once

#include "attn_block.cuh"
#include "bf16t_block.cuh"
#include "fp8_block.cuh"
#include "kv_quant.cuh"
#include "merge.cuh"
#include "paged_decode.cuh"
#include "pkv_split.cuh"

namespace pkv {

namespace {

// The decode's unit of work is a 16-token slice of a sequence (kBS tokens, a "unit"); a
// pool block of block_size tokens holds block_size / 16 units (block sizes 16, 32, 64) or
// half of one (block size 8: a unit's two halves come from two pool blocks).

// Blocks of KV the work item (virtual sequence) v contributes.
__device__ __forceinline__ int32_t item_blocks(const DecodeArgs &a, int v, bool report) {
    const int s = v / a.head_tiles;
    int32_t ctx = a.context_lens[s];
    if (a.query_start_loc) {
        const int32_t q0 = a.query_start_loc[s], q1 = a.query_start_loc[s + 1];
        if (q0 < 0 || q1 < q0 || q1 > a.total_q) {
            if (report) flag_error(a.err, PKV_DEVERR_QUERY_LEN);
            return 0;
        }
        if (q1 - q0 != 1) return 0;  // a prefill chunk (other kernel) or no rows
        if (ctx < 1) {
            if (report) flag_error(a.err, PKV_DEVERR_QUERY_LEN);
            return 0;
        }
    }
    if (ctx < 0 || (int64_t)ctx > (int64_t)a.max_blocks_per_seq * a.block_size) {
        if (report) flag_error(a.err, PKV_DEVERR_CONTEXT_LEN);
        return 0;
    }
    return (ctx + kBS - 1) / kBS;
}

// Exclusive prefix sum of item_blocks over all items, into pre[0..V] (pre[V] = total).
__device__ void build_prefix(const DecodeArgs &a, int V, int32_t *pre, int32_t *scan_tmp, bool report) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (V + nt - 1) / nt;
    const int beg = min(V, tid * per), end = min(V, beg + per);
    int32_t local = 0;
    for (int v = beg; v < end; ++v) local += item_blocks(a, v, report);
    // inclusive warp scan
    const int lane = tid & 31, warp = tid >> 5;
    int32_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scan_tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = (nt + 31) >> 5;
        int32_t w = lane < nw ? scan_tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) scan_tmp[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    int32_t run = x - local + (warp > 0 ? scan_tmp[warp - 1] : 0);
    for (int v = beg; v < end; ++v) {
        pre[v] = run;
        run += item_blocks(a, v, false);
    }
    if (tid == nt - 1) pre[V] = run;
    __syncthreads();
}

// Largest v in [0, V) with pre[v] <= f, for 0 <= f < pre[V].
__device__ __forceinline__ int find_item(const int32_t *pre, int V, int64_t f) {
    int lo = 0, hi = V;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= f) lo = mid; else hi = mid;
    }
    return lo;
}

// Unit f moved back to the first unit of its item (T stays T): with every share boundary
// moved so, each item lies whole in the share holding its first unit.
__device__ __forceinline__ int64_t item_floor(const int32_t *pre, int V, int64_t T, int64_t f) {
    return f >= T ? T : (int64_t)pre[find_item(pre, V, f)];
}

}  // namespace

// CTA 0: one merge job per boundary between CTA shares (the item split there, when that
// is its first split), and zero rows for decode rows whose context is empty.
template <int D>
__device__ void write_jobs_and_empty_rows(const DecodeArgs &a, const int32_t *pre, int V, int64_t T,
                                          int ge) {
    const int rows = a.heads_per_cta * a.group;
    for (int b = threadIdx.x; b < a.grid; b += blockDim.x) {
        MergeJob j;
        no_job(j);
        if (T > 0 && b < ge - 1 && !a.whole_items) {
            const int64_t f = share_begin(b + 1, T, ge);
            const int v = find_item(pre, V, f);
            const int64_t item_beg = pre[v];
            if (item_beg != f && item_beg >= share_begin(b, T, ge)) {
                const int s = v / a.head_tiles, ht = v - s * a.head_tiles;
                j.item_begin = item_beg;
                j.total_units = T;
                j.out_row0 = a.query_start_loc ? a.query_start_loc[s] : s;
                j.c0 = b;
                j.c1 = share_owner(pre[v + 1] - 1, T, ge);
                j.ge = ge;
                j.rows = rows;
                j.rows_per_token = rows;
                j.head0 = ht * rows;
            }
        }
        a.ws_jobs[b] = j;
    }
    const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int v = w; v < V; v += nw) {  // one warp per empty item
        if (pre[v] != pre[v + 1]) continue;
        const int s = v / a.head_tiles, ht = v - s * a.head_tiles;
        int64_t qrow = s;
        if (a.query_start_loc) {
            const int32_t q0 = a.query_start_loc[s], q1 = a.query_start_loc[s + 1];
            if (q1 - q0 != 1 || q0 < 0 || q1 > a.total_q) continue;
            qrow = q0;
        }
        __nv_bfloat16 *orow = a.out + (qrow * a.num_heads + (int64_t)ht * rows) * D;
        for (int i = lane; i < rows * D / 2; i += 32) reinterpret_cast<uint32_t *>(orow)[i] = 0u;
    }
}

// One CTA of the decode: CTA `cta` of `grid_eff` CTAs sharing the decode work (the
// whole grid for paged_decode_kernel; the decode CTAs of a varlen launch).  Merge jobs
// are written for all a.grid job slots (a.grid >= grid_eff).  `pdl`: wait for the
// previous kernel here (false when the caller already did).
// FP8: the cache holds e4m3 codes (head_dim 128 only); see fp8_block.cuh.  NTH: n-tiles of
// 8 query heads per consumer warp (1: a KV head has at most 8 query heads, else 2).
template <int D, bool FP8, int NTH>
__device__ __forceinline__ void decode_cta(const CUtensorMap &k_map, const CUtensorMap &v_map,
                                           const DecodeArgs &a, const int cta, const int grid_eff,
                                           const bool pdl) {
    static_assert(!FP8 || D == 128, "the FP8 cache path is built for head_dim 128");
    constexpr int KSTEPS = D / 16;         // k-steps of the QK^T MMA
    constexpr int DCH = FP8 ? 1 : D / 64;  // TMA boxes per block row (128 bytes each)

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int HT = a.heads_per_cta;
    const int NST = a.num_stages;
    const uint32_t stage_bytes = (uint32_t)HT * D * kBS * (FP8 ? 1 : 2);
    const uint32_t chunk_stride = (uint32_t)HT * kBS * 128;  // between 64-column sub-tiles
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NST * stage_bytes);
    uint64_t *empty = full + NST;
    int32_t *scan_tmp = reinterpret_cast<int32_t *>(empty + NST);  // 32 ints
    volatile int *abort_flag = scan_tmp + 32;
    int32_t *pre = scan_tmp + 36;

    const int V = a.num_seqs * a.head_tiles;
    const int ncw = HT * a.warps_per_head;  // consumer warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], ncw);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32 * ncw) {
        tma_prefetch_desc(&k_map);
        tma_prefetch_desc(&v_map);
    }
    // Everything above overlaps the previous kernel; from here on we read its output.
    if (pdl) {
        pdl_wait();
        pdl_trigger();
    }
    build_prefix(a, V, pre, scan_tmp, cta == 0);  // ends with __syncthreads
    const int64_t T = pre[V];
    const int ge = split_ctas(T, grid_eff, a.min_blocks_per_cta);
    if (cta == 0) write_jobs_and_empty_rows<D>(a, pre, V, T, ge);
    if (cta >= ge || T == 0) return;
    const int c = cta;
    int64_t lo = share_begin(c, T, ge), hi = share_begin(c + 1, T, ge);
    if (a.whole_items) {  // the split-K ablation: no partial items, no merge jobs
        lo = item_floor(pre, V, T, lo);
        hi = item_floor(pre, V, T, hi);
    }

    if (warp == ncw) {
        // ------------------------------ producer ------------------------------
        const uint64_t policy = l2_policy_evict_first();
        uint32_t stage = 0, phase = 0;
        uint32_t issued = 0;
        bool ok = true;
        const int bsz = a.block_size;
        auto checked = [&](int id) {
            if (id < 0 || (int64_t)id >= a.num_blocks) {
                flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                return -1;  // TMA fills the out-of-range box with zeros
            }
            return id;
        };
        const int Hkv = a.num_heads / a.group;
        for (int64_t f0 = lo; f0 < hi && ok; f0 += 32) {
            const int64_t f = f0 + lane;
            int bid = -1, bid2 = -1, ht = 0, tok0 = 0;
            int64_t wslot = -1;  // fused KV write: slot of the new token if this is its unit
            int wseq = 0;
            if (f < hi) {
                const int v = find_item(pre, V, f);
                const int s = v / a.head_tiles;
                ht = v - s * a.head_tiles;
                const int lb = (int)(f - pre[v]);  // unit inside the sequence
                const int32_t *row = a.block_tables + (int64_t)s * a.max_blocks_per_seq;
                if (a.k_new && f == pre[v + 1] - 1) {
                    const int p = a.context_lens[s] - 1;  // the new token's position
                    const int nb = checked(row[p / bsz]);
                    if (nb >= 0) {
                        wslot = (int64_t)nb * bsz + p % bsz;
                        wseq = s;
                        // pull the new rows into L2 now: the copy below runs when the unit
                        // comes up, up to 32 units later
                        const int64_t src = ((int64_t)s * Hkv + (int64_t)ht * HT) * D * 2;
                        const char *kp = static_cast<const char *>(a.k_new) + src;
                        const char *vp = static_cast<const char *>(a.v_new) + src;
                        for (int off = 0; off < HT * D * 2; off += 128) {
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(kp + off));
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(vp + off));
                        }
                    }
                }
                if (bsz >= kBS) {
                    const int r = bsz / kBS;
                    bid = checked(row[lb / r]);
                    tok0 = (lb % r) * kBS;
                } else {  // 8-token blocks: the unit's second half exists only inside the context
                    bid = checked(row[2 * lb]);
                    if (2 * lb + 1 < (a.context_lens[s] + bsz - 1) / bsz) bid2 = checked(row[2 * lb + 1]);
                }
            }
            const int n = (int)min64(32, hi - f0);
            for (int j = 0; j < n; ++j) {
                const int b = __shfl_sync(0xffffffffu, bid, j);
                const int b2 = __shfl_sync(0xffffffffu, bid2, j);
                const int t = __shfl_sync(0xffffffffu, ht, j);
                const int tk = __shfl_sync(0xffffffffu, tok0, j);
                const int64_t ws = __shfl_sync(0xffffffffu, wslot, j);
                if (ws >= 0) {
                    // The unit holds its sequence's new token: store the token's K and V rows
                    // for this item's heads (the whole warp), then order those stores before
                    // the TMA reads of the unit (async proxy) issued below.
                    const int sj = __shfl_sync(0xffffffffu, wseq, j);
                    const int64_t dst_off = ws * Hkv + (int64_t)t * HT;   // in head rows
                    const int64_t src_off = (int64_t)sj * Hkv + (int64_t)t * HT;
                    if constexpr (FP8) {
                        constexpr int V16 = D / 16;  // 16-code vectors per head row
                        const uint4 *ks = reinterpret_cast<const uint4 *>(a.k_new) + src_off * (D / 8);
                        const uint4 *vs = reinterpret_cast<const uint4 *>(a.v_new) + src_off * (D / 8);
                        uint4 *kd = reinterpret_cast<uint4 *>(a.k_cache_w) + dst_off * V16;
                        uint4 *vd = reinterpret_cast<uint4 *>(a.v_cache_w) + dst_off * V16;
                        for (int i = lane; i < HT * V16; i += 32) {
                            const uint4 k0 = ks[2 * i], k1 = ks[2 * i + 1];
                            const uint4 v0 = vs[2 * i], v1 = vs[2 * i + 1];
                            kd[i] = make_uint4(e4m3x4_of(k0.x, k0.y, a.k_scale_q), e4m3x4_of(k0.z, k0.w, a.k_scale_q),
                                               e4m3x4_of(k1.x, k1.y, a.k_scale_q), e4m3x4_of(k1.z, k1.w, a.k_scale_q));
                            vd[i] = make_uint4(e4m3x4_of(v0.x, v0.y, a.v_scale_q), e4m3x4_of(v0.z, v0.w, a.v_scale_q),
                                               e4m3x4_of(v1.x, v1.y, a.v_scale_q), e4m3x4_of(v1.z, v1.w, a.v_scale_q));
                        }
                    } else {
                        constexpr int V8 = D / 8;  // 16-byte vectors per head row
                        const uint4 *ks = reinterpret_cast<const uint4 *>(a.k_new) + src_off * V8;
                        const uint4 *vs = reinterpret_cast<const uint4 *>(a.v_new) + src_off * V8;
                        uint4 *kd = reinterpret_cast<uint4 *>(a.k_cache_w) + dst_off * V8;
                        uint4 *vd = reinterpret_cast<uint4 *>(a.v_cache_w) + dst_off * V8;
                        for (int i = lane; i < HT * V8; i += 32) {
                            kd[i] = ks[i];
                            vd[i] = vs[i];
                        }
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __syncwarp();
                }
                if (lane == 0) {
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.wait_ns)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[stage], stage_bytes);
                        uint8_t *dst = smem + (size_t)stage * stage_bytes;
                        const CUtensorMap *map = kv == 0 ? &k_map : &v_map;
                        if (bsz >= kBS) {
#pragma unroll
                            for (int dc = 0; dc < DCH; ++dc)
                                tma_load_5d(dst + dc * chunk_stride, map, &full[stage], 0, tk, t * HT,
                                            dc, b, policy);
                        } else {
                            // one 8-token box per head and half: each head's 16 rows stay
                            // contiguous (the swizzle follows the shared-memory address)
                            for (int dc = 0; dc < DCH; ++dc)
                                for (int h = 0; h < HT; ++h)
                                    for (int half = 0; half < 2; ++half)
                                        tma_load_5d(dst + dc * chunk_stride + h * (kBS * 128) + half * (8 * 128),
                                                    map, &full[stage], 0, 0, t * HT + h, dc, half ? b2 : b,
                                                    policy);
                        }
                        ++issued;
                        if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1; }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
        }
        if (!ok && lane == 0) {
            flag_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
            // Let the copies already issued land before the CTA's shared memory goes away.
            const uint32_t pending = minu32(issued, (uint32_t)NST);
            uint32_t st = stage, ph = phase;
            for (uint32_t i = 0; i < pending; ++i) {
                if (st == 0) { st = NST; ph ^= 1; }
                --st;
                mbar_wait(&full[st], ph, nullptr);
            }
        }
        return;
    }
    if (warp > ncw) return;

    // -------------------------------- consumers --------------------------------
    // Both caches put the group's query heads on the MMA's N and the block's 16 tokens on
    // M (S^T = K Q^T, O^T += V^T P^T): bf16t_block.cuh for bf16, fp8_block.cuh for e4m3.
    const int hh = warp / a.warps_per_head;                 // KV head inside the tile
    const int r0 = (warp - hh * a.warps_per_head) * 16;     // first query head of the warp
    const int g_row = lane >> 2, q4 = lane & 3;
    const int group = a.group;
    const uint32_t smem_base = smem_u32(smem);
    const float sl2 = a.scale_log2;

    uint32_t stage = 0, phase = 0;
    int64_t f = lo;
    HeadState<NTH> hs;
    while (f < hi) {
        const int v = find_item(pre, V, f);
        const int s = v / a.head_tiles;
        const int ht = v - s * a.head_tiles;
        const int64_t item_beg = pre[v], item_end = pre[v + 1];
        const int64_t seg_end = min64(hi, item_end);
        const int ctx = a.context_lens[s];
        const int64_t qrow = a.query_start_loc ? a.query_start_loc[s] : s;
        const int kvh = ht * HT + hh;
        const int rows_valid = min(16, group - r0);  // query heads this warp owns
        const __nv_bfloat16 *qw = a.q + (qrow * a.num_heads + (int64_t)kvh * group + r0) * D;

        // Q fragments: the FP8 form's A operand in its k numbering, or Q^T as the B operand
        uint32_t qa[FP8 ? KSTEPS : 1][4];
        uint32_t qb[FP8 ? 1 : NTH][FP8 ? 1 : KSTEPS][2];
        if constexpr (FP8) load_q_fp8order(qa, qw, rows_valid, lane);
        else load_q_bt<D, NTH>(qb, qw, rows_valid, lane);
        hs.reset();

        bool ok = true;
        for (; f < seg_end; ++f) {
            const int lb = (int)(f - item_beg);
            const int valid = min(kBS, ctx - lb * kBS);
            // ---- S^T = K Q^T over the block's 16 tokens ----
            if (!mbar_wait(&full[stage], phase, abort_flag, a.wait_ns)) { ok = false; break; }
            float sacc[NTH][4];
            const uint32_t ktile = smem_base + stage * stage_bytes + hh * (kBS * 128);
            if constexpr (FP8) qk_block_fp8t<NTH>(sacc, qa, ktile, lane);
            else qk_block_bt<D, NTH>(sacc, qb, ktile, chunk_stride, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1; }

            // ---- scale, mask the block's tail, online softmax (base 2) ----
            // S^T: tokens g (entries 0, 1) and g + 8 (entries 2, 3) of each n-tile
            const bool tail = valid < kBS;  // only a sequence's last block
            const bool in0 = !tail || g_row < valid, in1 = !tail || g_row + 8 < valid;
            uint32_t pb[NTH][2];
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) {
                sacc[nt][0] = in0 ? sacc[nt][0] * sl2 : -INFINITY;
                sacc[nt][1] = in0 ? sacc[nt][1] * sl2 : -INFINITY;
                sacc[nt][2] = in1 ? sacc[nt][2] * sl2 : -INFINITY;
                sacc[nt][3] = in1 ? sacc[nt][3] * sl2 : -INFINITY;
                if constexpr (FP8) softmax_update_t(hs, nt, sacc[nt], pb[nt]);
                else softmax_update_bt(hs, nt, sacc[nt], pb[nt]);
            }
            // ---- O^T += V^T P^T ----
            if (!mbar_wait(&full[stage], phase, abort_flag, a.wait_ns)) { ok = false; break; }
            const uint32_t vtile = smem_base + stage * stage_bytes + hh * (kBS * 128);
            if constexpr (FP8) {
                if (tail) pv_block_fp8t<true>(hs, pb, vtile, valid, lane);
                else pv_block_fp8t<false>(hs, pb, vtile, valid, lane);
            } else {
                if (tail) pv_block_bt<D, true>(hs, pb, vtile, chunk_stride, valid, lane);
                else pv_block_bt<D, false>(hs, pb, vtile, chunk_stride, valid, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1; }
        }
        if (!ok) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
            return;
        }

        // ---- finish this item's part ----
        const int64_t seg_beg = max64(lo, item_beg);
        const bool whole = seg_beg == item_beg && seg_end == item_end;
        finish_sums_t(hs);
        const float vs = a.v_scale;  // FP8: V elements are code x v_scale (1 for bf16)
        const int rows = HT * group;
        const int row0 = hh * group + r0;  // row inside the item
        const int slot = whole ? 0 : part_slot(c, item_beg, T, ge);
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int hd = 8 * nt + 2 * q4 + e;  // head inside the warp's 16
                if (hd >= rows_valid) continue;
                if constexpr (FP8) {
                    // lane (g, t) holds dims 16g .. 16g + 15: dim 16g + 2mt in o[nt][mt][e],
                    // 16g + 2mt + 1 in o[nt][mt][2 + e]
                    if (whole) {
                        const float inv = vs / hs.l[nt][e];
                        uint32_t p[8];
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt)
                            p[mt] = pack_bf16x2(hs.o[nt][mt][e] * inv, hs.o[nt][mt][2 + e] * inv);
                        uint4 *orow = reinterpret_cast<uint4 *>(
                            a.out + (qrow * a.num_heads + (int64_t)kvh * group + r0 + hd) * D + 16 * g_row);
                        orow[0] = make_uint4(p[0], p[1], p[2], p[3]);
                        orow[1] = make_uint4(p[4], p[5], p[6], p[7]);
                    } else {
                        float4 *ob = reinterpret_cast<float4 *>(a.ws_o + ((int64_t)slot * rows + row0 + hd) * D +
                                                                16 * g_row);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            ob[k] = make_float4(hs.o[nt][2 * k][e] * vs, hs.o[nt][2 * k][2 + e] * vs,
                                                hs.o[nt][2 * k + 1][e] * vs, hs.o[nt][2 * k + 1][2 + e] * vs);
                    }
                } else {
                    // lane (g, t) holds dims 16mt + g (o[nt][mt][e]) and 16mt + g + 8 (o[nt][mt][2 + e])
                    if (whole) {
                        const float inv = 1.f / hs.l[nt][e];
                        __nv_bfloat16 *orow = a.out + (qrow * a.num_heads + (int64_t)kvh * group + r0 + hd) * D;
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            orow[16 * mt + g_row] = __float2bfloat16_rn(hs.o[nt][mt][e] * inv);
                            orow[16 * mt + g_row + 8] = __float2bfloat16_rn(hs.o[nt][mt][2 + e] * inv);
                        }
                    } else {
                        float *ob = a.ws_o + ((int64_t)slot * rows + row0 + hd) * D;
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            ob[16 * mt + g_row] = hs.o[nt][mt][e];
                            ob[16 * mt + g_row + 8] = hs.o[nt][mt][2 + e];
                        }
                    }
                }
                if (!whole && g_row == 0)
                    a.ws_ml[(int64_t)slot * rows + row0 + hd] = make_float2(hs.m[nt][e], hs.l[nt][e]);
            }
        f = seg_end;
    }
}

}  // namespace pkv
