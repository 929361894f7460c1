// prefill_cta.cuh -- one CTA's share of the chunked-prefill attention over a block-paged
// KV cache (the body of paged_prefill_kernel, also run by the prefill CTAs of
// paged_varlen_kernel).
//
// Method: "Servis Motor İçleri: PagedAttention, Sürekli Batching, parçalanmış Prefill"
// (aiengineeringfromscratch.com, Phase 17 - 04), "Chunked prefill protects the TTFT
// tail": a long prompt is cut into fixed-size chunks (512 tokens by default) and each
// chunk runs as one unit of an iteration's batch, next to single-token decodes.  A
// chunk's queries are the last q_len positions of its sequence's context, so with
// causal masking row j sees keys 0 .. context_len - q_len + j: its paged prefix and
// the chunk up to itself.  Keys are found through the block table as in
// "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn), §2.3.
//
// GB300 design
//  * A tile is 2 halves x (16 * 8 / group) query tokens x the `group` query heads of one
//    KV head, i.e. two 128-row tcgen05 MMA tiles for Llama-70B shapes; both halves use
//    every K/V chunk in shared memory, so a key is read from L2 once per 256 query rows.
//  * Keys go in 128-key chunks (8 blocks).  One elected thread issues S = Q K^T
//    (128 x 128 x head_dim, A and B from 128-byte-swizzled shared memory) into TMEM, the
//    half's softmax warpgroup (one thread per row) reads the row's 128 scores once (two
//    64-column TMEM loads that also return their maximum), writes the bf16 weights P
//    back over S, and O += P V runs with P as the A operand straight from TMEM.  The halves alternate on the tensor pipe, so one
//    half's MMAs overlap the other half's softmax.  Online softmax in base 2, rescaled
//    only when a row's maximum grows by more than 2^8 (O is then rescaled in TMEM).
//  * The units are (tile, 16-token key block) pairs; causal tiles stop at the block
//    holding their last query's position.  A persistent grid (one CTA per SM) takes
//    equal contiguous shares of the flat unit list, so long prefixes split across
//    CTAs and no SM idles in a tail; split tiles are merged by log-sum-exp weights.
//  * A producer warp streams K and V of each chunk with TMA (one 5-D box per block and
//    64-column slice) into a ring of shared-memory stages.
//  * Waits are bounded in time; no CTA waits on another CTA.
#pragma once

#include "attn_block.cuh"
#include "fp32x2.cuh"
#include "fp8_block.cuh"
#include "merge.cuh"
#include "paged_prefill.cuh"
#include "pkv_split.cuh"
#include "tcgen05.cuh"


namespace pkv {

namespace {


// Closed forms for one sequence's tiles.  Tile qt covers query tokens
// [qt*TPT, min(q_len, (qt+1)*TPT)).  Causal: the tile visits key blocks
// 0 .. ceil((pos_last + 1) / 16) - 1; with TPT a multiple of 16 a full tile qt visits
// A + (qt + 1) * B blocks, A = ceil((ctx - q_len) / 16), B = TPT / 16.
struct SeqTiles {
    int ctx, q_len, q_row0;
    int64_t A, B, nfull, rem, nk_all;  // nk_all = ceil(ctx / 16)
    bool causal;
    int64_t per_head;                  // units of one KV head: sum over tiles

    // units before tile qt (qt <= nfull)
    __device__ __forceinline__ int64_t before(int64_t qt) const {
        return causal ? qt * A + B * qt * (qt + 1) / 2 : qt * nk_all;
    }
    __device__ __forceinline__ int64_t blocks_of(int64_t qt) const {
        return (!causal || qt >= nfull) ? nk_all : A + (qt + 1) * B;
    }
    // tile holding unit o1 of one head (0 <= o1 < per_head)
    __device__ __forceinline__ int64_t tile_of(int64_t o1) const {
        if (o1 >= before(nfull)) return nfull;
        int64_t lo = 0, hi = nfull;
        while (hi - lo > 1) {
            const int64_t mid = (lo + hi) >> 1;
            if (before(mid) <= o1) lo = mid; else hi = mid;
        }
        return lo;
    }
};

// Reads sequence s; returns false if it has no prefill rows (q_len < 2) or invalid
// metadata (flagged when `report`).
__device__ __forceinline__ bool seq_tiles(const PrefillArgs &a, int s, bool report, SeqTiles &t) {
    const int32_t q0 = a.query_start_loc[s], q1 = a.query_start_loc[s + 1];
    const int32_t ql = q1 - q0;
    if (q0 < 0 || ql < 0 || q1 > a.total_q) {
        if (report) flag_error(a.err, PKV_DEVERR_QUERY_LEN);
        return false;
    }
    if (ql < 2) return false;
    const int32_t ctx = a.context_lens[s];
    if (ctx < 0 || (int64_t)ctx > (int64_t)a.max_blocks_per_seq * kBS) {
        if (report) flag_error(a.err, PKV_DEVERR_CONTEXT_LEN);
        return false;
    }
    if (ql > ctx) {
        if (report) flag_error(a.err, PKV_DEVERR_QUERY_LEN);
        return false;
    }
    const int TPT = a.tokens_per_tile;
    t.ctx = ctx;
    t.q_len = ql;
    t.q_row0 = q0;
    t.causal = a.causal;
    t.A = (ctx - ql + kBS - 1) / kBS;
    t.B = TPT / kBS;
    t.nfull = ql / TPT;
    t.rem = ql % TPT;
    t.nk_all = (ctx + kBS - 1) / kBS;
    t.per_head = t.before(t.nfull) + (t.rem > 0 ? t.blocks_of(t.nfull) : 0);
    return true;
}

__device__ __forceinline__ int64_t seq_units(const PrefillArgs &a, int s, bool report) {
    SeqTiles t;
    if (!seq_tiles(a, s, report, t)) return 0;
    return t.per_head * a.num_kv_heads;
}

// pre[0..S] = units before each sequence (pre[S] = total), built by the whole CTA.
__device__ void build_seq_prefix(const PrefillArgs &a, int64_t *pre, int64_t *scan_tmp, bool report) {
    const int S = a.num_seqs;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (S + nt - 1) / nt;
    const int beg = min(S, tid * per), end = min(S, beg + per);
    int64_t local = 0;
    for (int s = beg; s < end; ++s) local += seq_units(a, s, report);
    const int lane = tid & 31, warp = tid >> 5;
    int64_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scan_tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = (nt + 31) >> 5;
        int64_t w = lane < nw ? scan_tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) scan_tmp[lane] = w;
    }
    __syncthreads();
    int64_t run = x - local + (warp > 0 ? scan_tmp[warp - 1] : 0);
    for (int s = beg; s < end; ++s) {
        pre[s] = run;
        run += seq_units(a, s, false);
    }
    if (tid == nt - 1) pre[S] = run;
    __syncthreads();
}

// Where unit f lives: sequence, KV head, tile, key block, and the tile's first unit.
struct UnitPos {
    int s, kvh;
    int64_t qt, kb, tile_begin, tile_blocks;
    SeqTiles t;
};

__device__ __forceinline__ void locate(const PrefillArgs &a, const int64_t *pre, int64_t f,
                                       UnitPos &u) {
    int lo = 0, hi = a.num_seqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= f) lo = mid; else hi = mid;
    }
    u.s = lo;
    seq_tiles(a, lo, false, u.t);
    const int64_t o = f - pre[lo];
    u.kvh = (int)(o / u.t.per_head);
    const int64_t o1 = o - (int64_t)u.kvh * u.t.per_head;
    u.qt = u.t.tile_of(o1);
    u.kb = o1 - u.t.before(u.qt);
    u.tile_begin = f - u.kb;
    u.tile_blocks = u.t.blocks_of(u.qt);
}

}  // namespace

// CTA 0: one merge job per boundary between CTA shares (the tile split there, when
// that is its first split), and zero rows for prefill sequences whose metadata was
// invalid (their units were dropped from the split).
template <int D>
__device__ void write_jobs_and_invalid_rows(const PrefillArgs &a, const int64_t *pre, int64_t T,
                                            int ge) {
    for (int b = threadIdx.x; b < a.grid; b += blockDim.x) {
        MergeJob j;
        no_job(j);
        if (T > 0 && b < ge - 1) {
            const int64_t f = share_begin(b + 1, T, ge);
            UnitPos u;
            locate(a, pre, f, u);
            if (u.kb != 0 && u.tile_begin >= share_begin(b, T, ge)) {
                j.item_begin = u.tile_begin;
                j.total_units = T;
                j.out_row0 = u.t.q_row0 + u.qt * a.tokens_per_tile;
                j.c0 = b;
                j.c1 = share_owner(u.tile_begin + u.tile_blocks - 1, T, ge);
                j.ge = ge;
                j.rows = (int)min64(a.tokens_per_tile, u.t.q_len - u.qt * a.tokens_per_tile) * a.group;
                j.rows_per_token = a.group;
                j.head0 = u.kvh * a.group;
            }
        }
        a.ws_jobs[b] = j;
    }
    const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int s = w; s < a.num_seqs; s += nw) {  // one warp per dropped sequence
        const int32_t q0 = a.query_start_loc[s], q1 = a.query_start_loc[s + 1];
        if (q1 - q0 < 2 || q0 < 0 || q1 > a.total_q || pre[s + 1] != pre[s]) continue;
        uint32_t *o = reinterpret_cast<uint32_t *>(a.out + (int64_t)q0 * a.num_heads * D);
        for (int64_t i = lane; i < (int64_t)(q1 - q0) * a.num_heads * D / 2; i += 32) o[i] = 0u;
    }
}

// Layout of the kernel's shared memory (offsets from a 1024-byte-aligned base).  A work
// tile is two halves of up to 128 query rows (one tcgen05 MMA M each); both halves use
// every K/V chunk the producer loads.
template <int D>
struct PrefillSmem {
    static constexpr int KT = 128;                             // keys per chunk (the QK MMA's N)
    static constexpr int BPC = KT / kBS;                       // blocks per chunk
    static constexpr uint32_t HALF_DC = 128 * 128;             // 128 rows x 64 columns of Q
    static constexpr uint32_t Q_DC = 2 * HALF_DC;              // both halves, one column chunk
    static constexpr uint32_t Q_BYTES = (D / 64) * Q_DC;
    static constexpr uint32_t KV_DC = KT * 128;                // 128 keys x 64 columns
    static constexpr uint32_t STG = (D / 64) * KV_DC;          // K or V of one chunk
    // Epilogue staging: 4 KiB per softmax warp (32 rows x 128 bytes), so O leaves in
    // whole 128-byte lines instead of one row per thread.
    static constexpr uint32_t EPI_WARP = 4096;
    static constexpr uint32_t OFF_EPI = Q_BYTES;
    static constexpr uint32_t OFF_STAGES = Q_BYTES + 8 * EPI_WARP;
    // TMEM, per half: S (128 fp32 columns; P overwrites its first 64 as bf16 pairs), O.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t HALF_COLS = 256;
    static constexpr uint32_t COL_O = 128;
};

// The CTA's share is walked segment by segment (a segment = the part of one tile that
// lies in the share); each segment's blocks go in chunks of up to BPC.
struct Segment {
    UnitPos u;
    int64_t end;     // one past the segment's last unit
    int nblk;        // blocks in the segment
    int chunks;      // ceil(nblk / BPC)
    int tile_tokens; // query tokens of the tile
};

template <int BPC>
__device__ __forceinline__ void segment_at(const PrefillArgs &a, const int64_t *pre, int64_t f,
                                           int64_t hi, Segment &sg) {
    locate(a, pre, f, sg.u);
    sg.end = min64(hi, sg.u.tile_begin + sg.u.tile_blocks);
    sg.nblk = (int)(sg.end - f);
    sg.chunks = (sg.nblk + BPC - 1) / BPC;
    sg.tile_tokens = (int)min64(a.tokens_per_tile, sg.u.t.q_len - sg.u.qt * a.tokens_per_tile);
}

// FP8: the cache holds e4m3 codes (head_dim 128).  The producer loads them into a ring of
// byte stages; warps 2 and 3 widen each chunk to fp16 into the operand ring the MMAs read
// (same swizzled layout as the bf16 path), zero V rows past the context, and convert each
// tile's Q to fp16 in place; the MMAs run kind::f16 with fp16 operands and P is fp16.
// One CTA of the chunked prefill: CTA `cta` of `grid_eff` CTAs sharing the prefill work
// (the whole grid for paged_prefill_kernel; the prefill CTAs of a varlen launch).  Merge
// jobs are written for all a.grid job slots (a.grid >= grid_eff).  `pdl`: wait for the
// previous kernel here (false when the caller already did).
template <int D, bool FP8>
__device__ __forceinline__ void prefill_cta(const CUtensorMap &q_map, const CUtensorMap &k_map,
                                            const CUtensorMap &v_map, const PrefillArgs &a,
                                            const int cta, const int grid_eff, const bool pdl) {
    static_assert(!FP8 || D == 128, "the FP8 prefill is built for head_dim 128");
    using L = PrefillSmem<D>;
    constexpr int DCH = D / 64;
    constexpr uint32_t IDESC_QK = FP8 ? umma_idesc_f16(128, L::KT, 0, 0) : umma_idesc_bf16(128, L::KT, 0, 0);
    constexpr uint32_t IDESC_PV = FP8 ? umma_idesc_f16(128, D, 0, 1) : umma_idesc_bf16(128, D, 0, 1);
    constexpr uint32_t STG8 = L::KT * D;  // e4m3 K or V of one chunk

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NST = a.num_stages;
    uint8_t *sQ = smem, *sStage = smem + L::OFF_STAGES, *sEpi = smem + L::OFF_EPI;
    const int NST8 = FP8 ? a.num_stages8 : 0;
    uint8_t *s8 = sStage + (size_t)NST * L::STG;  // FP8: the e4m3 staging ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(s8 + (size_t)NST8 * STG8);
    // per half h: s_full[h], p_full[h], pv_done[h], o_free[h]
    uint64_t *q_full = bars, *q_empty = bars + 1, *mma_done = bars + 2;
    uint64_t *s_full = bars + 3, *p_full = bars + 5, *pv_done = bars + 7, *o_free = bars + 9;
    uint64_t *kv_full = bars + 11, *kv_empty = kv_full + NST;
    // FP8: e4m3 stages landed / converted; Q of the segment converted to fp16
    uint64_t *f8_full = kv_empty + NST, *f8_empty = f8_full + NST8, *q_ready = f8_empty + NST8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(q_ready + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int64_t *scan_tmp = reinterpret_cast<int64_t *>(tmem_slot + 2);  // 32 entries
    int64_t *pre = scan_tmp + 32;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = a.group, TPT = a.tokens_per_tile, HTOK = TPT / 2;
    const int tile_rows = TPT * group, half_rows = HTOK * group;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(mma_done, 1);
        for (int h = 0; h < 2; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&p_full[h], 4);  // one arrival per softmax warp
            mbar_init(&pv_done[h], 1);
            mbar_init(&o_free[h], 4);
        }
        for (int i = 0; i < NST; ++i) {
            mbar_init(&kv_full[i], FP8 ? 64 : 1);  // FP8: the 64 converter threads arrive
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < NST8; ++i) {
            mbar_init(&f8_full[i], 1);
            mbar_init(&f8_empty[i], 64);
        }
        mbar_init(q_ready, 64);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&q_map);
        tma_prefetch_desc(&k_map);
        tma_prefetch_desc(&v_map);
    }
    if (pdl) {
        pdl_wait();
        pdl_trigger();
    }
    build_seq_prefix(a, pre, scan_tmp, cta == 0);  // ends with __syncthreads
    const int64_t T = pre[a.num_seqs];
    const int ge = split_ctas(T, grid_eff, 4);
    if (cta == 0) write_jobs_and_invalid_rows<D>(a, pre, T, ge);
    if (cta >= ge || T == 0) return;
    const int c = cta;
    const int64_t lo = share_begin(c, T, ge), hi = share_begin(c + 1, T, ge);

    if (warp == 1) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        const uint64_t policy = l2_policy_evict_normal();
        uint32_t fill = 0, pst = 0, pph = 0;  // copies issued; ring slot of the next one
        int seg_i = 0;
        bool ok = true;
        for (int64_t f = lo; f < hi && ok;) {
            Segment sg;
            segment_at<L::BPC>(a, pre, f, hi, sg);
            const UnitPos &u = sg.u;
            if (lane == 0) {
                if (seg_i > 0) ok = mbar_wait(q_empty, (seg_i - 1) & 1, abort_flag, a.wait_ns);
                if (ok) {
                    mbar_arrive_expect_tx(q_full, 2 * DCH * half_rows * 128);
                    const int tok0 = (int)(u.t.q_row0 + u.qt * TPT);
                    for (int h = 0; h < 2; ++h)
                        for (int dc = 0; dc < DCH; ++dc)
                            tma_load_4d(sQ + dc * L::Q_DC + h * L::HALF_DC, &q_map, q_full, 0, dc,
                                        u.kvh * group, tok0 + h * HTOK, policy);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            const int64_t trow = (int64_t)u.s * a.max_blocks_per_seq + u.kb;
            for (int b0 = 0; b0 < sg.nblk && ok; b0 += 32) {
                int bid = -1;
                if (b0 + lane < sg.nblk) {
                    bid = a.block_tables[trow + b0 + lane];
                    if (bid < 0 || (int64_t)bid >= a.num_blocks) {
                        flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                        bid = -1;  // TMA fills an out-of-range box with zeros
                    }
                }
                const int n32 = min(32, sg.nblk - b0);
                for (int cb = 0; cb < n32 && ok; cb += L::BPC) {
                    int ids[L::BPC];
#pragma unroll
                    for (int i = 0; i < L::BPC; ++i) {
                        const int v = __shfl_sync(0xffffffffu, bid, (cb + i) & 31);
                        ids[i] = cb + i < n32 ? v : -1;  // missing blocks load as zeros
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int kv = 0; kv < 2; ++kv) {
                            const uint32_t st = pst;
                            // FP8: the e4m3 staging ring (the converters fill the operand ring)
                            uint64_t *fb = FP8 ? &f8_full[st] : &kv_full[st];
                            uint64_t *eb = FP8 ? &f8_empty[st] : &kv_empty[st];
                            if (!mbar_wait(eb, pph ^ 1, abort_flag, a.wait_ns)) {
                                ok = false;
                                break;
                            }
                            if (++pst == (uint32_t)(FP8 ? NST8 : NST)) { pst = 0; pph ^= 1; }
                            const CUtensorMap *map = kv == 0 ? &k_map : &v_map;
                            if constexpr (FP8) {
                                mbar_arrive_expect_tx(fb, STG8);
                                uint8_t *dst = s8 + (size_t)st * STG8;  // [key][128 bytes], 128-byte swizzle
#pragma unroll
                                for (int i = 0; i < L::BPC; ++i)
                                    tma_load_5d(dst + i * (kBS * 128), map, fb, 0, 0, u.kvh, 0, ids[i], policy);
                            } else {
                                mbar_arrive_expect_tx(fb, L::STG);
                                uint8_t *dst = sStage + (size_t)st * L::STG;
#pragma unroll
                                for (int i = 0; i < L::BPC; ++i)
#pragma unroll
                                    for (int dc = 0; dc < DCH; ++dc)
                                        tma_load_5d(dst + dc * L::KV_DC + i * (kBS * 128), map, fb, 0, 0,
                                                    u.kvh, dc, ids[i], policy);
                            }
                            ++fill;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                }
            }
            f = sg.end;
            ++seg_i;
        }
        if (!ok && lane == 0) {
            flag_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
            // let issued copies land before shared memory is released
            const uint32_t nring = FP8 ? NST8 : NST;
            const uint32_t pending = minu32(fill, nring);
            for (uint32_t k = fill - pending; k < fill; ++k)
                mbar_wait(FP8 ? &f8_full[k % nring] : &kv_full[k % nring], (k / nring) & 1, nullptr);
            if (seg_i > 0) mbar_wait(q_full, (seg_i - 1) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        // Per half h, S lives in TMEM columns [h*256, h*256+128); the softmax writes the bf16
        // weights P back over its first 64 columns, and PV takes them as the A operand from
        // TMEM.  The halves alternate on the tensor pipe: PV_0(c), QK_0(c+1), PV_1(c),
        // QK_1(c+1), so one half's MMAs run while the other half's softmax works.  QK_h(c+1)
        // overwrites S_h right after PV_h(c) read P_h from it; MMAs of one thread run in issue
        // order, and the softmax learns both are done from the commit behind QK_h(c+1).
        // The whole warp runs this loop on warp-uniform values and one elected lane issues
        // (the same lane every time, so each commit covers every MMA before it); waits end
        // together for the warp (a timeout seen by any lane aborts all of them).
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, a.wait_ns));
        };
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint64_t dq0 = umma_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = umma_desc_sw128(smem_u32(sStage), 16, 1024);
        const uint64_t dv0 = umma_desc_sw128(smem_u32(sStage), L::KV_DC, 1024);
        constexpr uint32_t STG16 = L::STG >> 4;
        uint32_t kst = 0, kph = 0;  // ring slot of the next chunk's K
        uint32_t gh[2] = {0, 0};    // chunks each half has processed
        int segh[2] = {0, 0};       // segments each half has processed
        int seg_i = 0;
        bool ok = true;
        bool issued = false;
        auto adv = [&](uint32_t &st, uint32_t &ph) {
            if (++st == (uint32_t)NST) { st = 0; ph ^= 1; }
        };
        auto issue_qk = [&](int h, uint32_t kslot) {
            const uint64_t dk = dk0 + kslot * STG16;
            const uint64_t dq = dq0 + h * (L::HALF_DC >> 4);
            const uint32_t tS = tm + h * L::HALF_COLS;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t koff = ((ks / 4) * L::KV_DC + (ks % 4) * 32) >> 4;
                const uint32_t qoff = ((ks / 4) * L::Q_DC + (ks % 4) * 32) >> 4;
                umma_bf16_warp(tS, dq + qoff, dk + koff, IDESC_QK, ks > 0);
            }
            umma_commit_warp(&s_full[h]);
            issued = true;
        };
        for (int64_t f = lo; f < hi && ok;) {
            Segment sg;
            segment_at<L::BPC>(a, pre, f, hi, sg);
            const int chunks = __shfl_sync(0xffffffffu, sg.chunks, 0);
            const int nh = __shfl_sync(0xffffffffu, sg.tile_tokens > HTOK ? 2 : 1, 0);  // halves with rows
            if (!wait_all(FP8 ? q_ready : q_full, seg_i & 1)) { ok = false; break; }
            // chunk 0's K and V slots
            uint32_t ks_ = kst, kp_ = kph;
            uint32_t vs_ = kst, vp_ = kph;
            adv(vs_, vp_);
            kst = vs_;
            kph = vp_;
            adv(kst, kph);
            if (!wait_all(&kv_full[ks_], kp_)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (h < nh) issue_qk(h, ks_);
            umma_commit_warp(&kv_empty[ks_]);
            if (chunks == 1) umma_commit_warp(q_empty);
            for (int ch = 0; ch < chunks && ok; ++ch) {
                const bool more = ch + 1 < chunks;
                uint32_t nks = kst, nkp = kph;  // the next chunk's K and V slots
                uint32_t nvs = kst, nvp = kph;
                if (more) {
                    adv(nvs, nvp);
                    kst = nvs;
                    kph = nvp;
                    adv(kst, kph);
                }
                if (!wait_all(&kv_full[vs_], vp_)) { ok = false; break; }
                const uint64_t dv = dv0 + vs_ * STG16;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h >= nh) break;
                    const uint32_t gg = gh[h] + ch;
                    if (ch == 0 && segh[h] > 0 && !wait_all(&o_free[h], (segh[h] - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (!wait_all(&p_full[h], gg & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t tP = tm + h * L::HALF_COLS;
                    const uint32_t tO = tP + L::COL_O;
#pragma unroll
                    for (int ks = 0; ks < L::KT / 16; ++ks)
                        umma_bf16_tmem_a_warp(tO, tP + ks * 8, dv + ks * (2048 >> 4), IDESC_PV,
                                              !(ch == 0 && ks == 0));
                    umma_commit_warp(&pv_done[h]);
                    if (h == nh - 1) umma_commit_warp(&kv_empty[vs_]);  // V(c) read by every half
                    if (more) {
                        if (h == 0 && !wait_all(&kv_full[nks], nkp)) { ok = false; break; }
                        issue_qk(h, nks);
                        if (h == nh - 1) {
                            umma_commit_warp(&kv_empty[nks]);
                            if (ch + 1 == chunks - 1) umma_commit_warp(q_empty);
                        }
                    }
                }
                if (!ok) break;
                vs_ = nvs;
                vp_ = nvp;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (h < nh) {
                    gh[h] += chunks;
                    segh[h] += 1;
                }
            f = sg.end;
            ++seg_i;
        }
        if (!ok) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
        // every MMA the warp issued is finished before TMEM is released
        if (issued) {
            umma_commit_warp(mma_done);
            mbar_wait(mma_done, 0, nullptr);
        }
        __syncwarp();
    } else if (FP8 && (warp == 2 || warp == 3)) {
        // ------------------ FP8: e4m3 -> fp16 converters (64 threads) ------------------
        // They walk the same segments and chunks as the producer.  Per segment: once the
        // tile's Q (bf16) has landed, convert it to fp16 in place and signal q_ready.  Per K or
        // V chunk: wait for its e4m3 stage and a free operand slot, widen 128 keys x 128
        // columns into the slot's layout ([64-column chunk][key][128 bytes], chunk c of a row
        // at c ^ (key % 8)), zero V rows at or past the context (the pool may hold NaN codes
        // there), then release the e4m3 stage and mark the slot full.  Generic stores become
        // visible to the tensor core through fence.proxy.async before each arrive.
        const int ctid = threadIdx.x - 64;
        // Lanes 8q .. 8q+7 (one 128-byte phase of a 16-byte access) take 8 keys of the same
        // 16-code group: their loads (chunk c8 ^ key % 8) and stores (chunk 2 (c8 % 4) ^ key % 8,
        // and its pair) then hit 8 different bank groups.
        const int c_key = ctid & 7, c8 = ctid >> 3, k7 = c_key;
        const int cp = (c8 & 3) * 2;  // first 16-byte chunk of the pair in a 64-column row
        const uint32_t c_src = c_key * 128 + ((c8 ^ k7) << 4);
        const uint32_t c_dst = (c8 >> 2) * L::KV_DC + c_key * 128 + ((cp ^ k7) << 4);
        const int c_pair = (((cp + 1) ^ k7) - (cp ^ k7)) << 4;  // +-16: the pair's second chunk
        uint32_t s8i = 0, p8 = 0, s16 = 0, p16 = 0;
        int seg_i = 0;
        bool ok = true;
        for (int64_t f = lo; f < hi && ok;) {
            Segment sg;
            segment_at<L::BPC>(a, pre, f, hi, sg);
            if (!mbar_wait(q_full, seg_i & 1, abort_flag, a.wait_ns)) { ok = false; break; }
            uint4 *q4 = reinterpret_cast<uint4 *>(sQ);
#pragma unroll 8
            for (int i = ctid; i < (int)(L::Q_BYTES / 16); i += 64) {
                uint4 x = q4[i];
                x.x = bf16x2_to_f16x2(x.x);
                x.y = bf16x2_to_f16x2(x.y);
                x.z = bf16x2_to_f16x2(x.z);
                x.w = bf16x2_to_f16x2(x.w);
                q4[i] = x;
            }
            fence_async_smem();
            mbar_arrive(q_ready);
            const int ctx = sg.u.t.ctx;
            for (int ch = 0; ch < sg.chunks && ok; ++ch) {
                const int64_t key0 = (sg.u.kb + (int64_t)L::BPC * ch) * kBS;
#pragma unroll 1
                for (int kv = 0; kv < 2; ++kv) {
                    if (!mbar_wait(&f8_full[s8i], p8, abort_flag, a.wait_ns) || !mbar_wait(&kv_empty[s16], p16 ^ 1, abort_flag, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // Thread t always handles 16-code group c8 = t / 8 of keys t % 8 + 8 j (j < 16):
                    // key % 8 is fixed per thread, so the swizzled offsets are too, and the
                    // 16 steps differ by 1 KiB.  All 16 loads are issued before the first store
                    // (the compiler may not move a load above a store it cannot disambiguate),
                    // so the loop is not a chain of shared-memory round trips.
                    const uint8_t *src = s8 + (size_t)s8i * STG8 + c_src;
                    uint8_t *dst = sStage + (size_t)s16 * L::STG + c_dst;
                    const int zero_from = kv == 1 ? (int)max64(0, min64(ctx - key0, (int64_t)L::KT)) : L::KT;
                    uint4 x[L::KT / 8];
#pragma unroll
                    for (int j = 0; j < L::KT / 8; ++j) x[j] = *reinterpret_cast<const uint4 *>(src + j * 1024);
#pragma unroll
                    for (int j = 0; j < L::KT / 8; ++j) {
                        uint4 lo4, hi4;
                        e4m3x4_to_f16x2x2(x[j].x, lo4.x, lo4.y);
                        e4m3x4_to_f16x2x2(x[j].y, lo4.z, lo4.w);
                        e4m3x4_to_f16x2x2(x[j].z, hi4.x, hi4.y);
                        e4m3x4_to_f16x2x2(x[j].w, hi4.z, hi4.w);
                        if (c_key + 8 * j >= zero_from) lo4 = hi4 = make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(dst + j * 1024) = lo4;
                        *reinterpret_cast<uint4 *>(dst + j * 1024 + c_pair) = hi4;
                    }
                    fence_async_smem();
                    mbar_arrive(&kv_full[s16]);
                    mbar_arrive(&f8_empty[s8i]);
                    if (++s8i == (uint32_t)NST8) { s8i = 0; p8 ^= 1; }
                    if (++s16 == (uint32_t)NST) { s16 = 0; p16 ^= 1; }
                }
            }
            f = sg.end;
            ++seg_i;
        }
        if (!ok) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp >= 4) {
        // -------------- softmax: one warpgroup per half, one row per thread --------------
        const int h = (warp - 4) >> 2;
        const int quarter = warp & 3;  // the TMEM lanes this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t tl = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + tl + h * L::HALF_COLS;
        const uint32_t tO = tS + L::COL_O;
        const int tid = threadIdx.x - 128 - 128 * h;  // 0..127 within the warpgroup
        const float sl2 = a.scale_log2;
        uint32_t gh = 0;   // chunks this half has processed
        uint32_t gk = 0;   // chunks of the CTA (K/V ring position)
        bool ok = true;
        for (int64_t f = lo; f < hi && ok;) {
            Segment sg;
            segment_at<L::BPC>(a, pre, f, hi, sg);
            const UnitPos &u = sg.u;
            if (h == 1 && sg.tile_tokens <= HTOK) {  // this half has no query rows here
                gk += sg.chunks;
                f = sg.end;
                continue;
            }
            const int ctx = u.t.ctx;
            const int half_tokens = min(HTOK, sg.tile_tokens - h * HTOK);
            const int tok_l = row / group, hg = row - tok_l * group;
            const bool rvalid = row < half_rows && tok_l < half_tokens;
            const int tok = h * HTOK + tok_l;  // token inside the tile
            const int64_t first_pos = (int64_t)(ctx - u.t.q_len) + u.qt * TPT;
            const int64_t lim =
                a.causal ? min64(first_pos + min(tok, sg.tile_tokens - 1) + 1, ctx) : ctx;
            float m_ref = -INFINITY, l = 0.f;
            for (int ch = 0; ch < sg.chunks; ++ch, ++gh, ++gk) {
                const int nb = min(L::BPC, sg.nblk - L::BPC * ch);
                const int64_t key0 = (u.kb + (int64_t)L::BPC * ch) * kBS;
                const int nkeys = nb * kBS;
                if (!mbar_wait(&s_full[h], gh & 1, abort_flag, a.wait_ns)) { ok = false; break; }
                tc_fence_after();
                // visible keys of this chunk for this row: [0, vis)
                const int vis = (int)max64(0, min64(lim - key0, (int64_t)nkeys));
                const bool full = __all_sync(0xffffffffu, vis >= L::KT);
                // One pass over the row's 128 scores in two rounds of 64 columns.  A round's
                // loads also return its maximum (tcgen05.ld.red); the weights are taken
                // against the row's reference maximum m_ref, which moves (lazy rescale) only
                // when a round's maximum exceeds it by more than kRescaleSlack.  A move in the
                // second round rescales the first round's weights, already in TMEM, and any
                // move rescales O (both after the weights, when the scores' registers are free).
                // A chunk with keys a row may not see (causal diagonal, context end) masks
                // them before an ALU maximum instead.
                float a_o = 1.f, a_p0 = 1.f;   // this chunk's scale of O / of round 0's weights
                bool any_o = false, any_p0 = false;
                uint64_t ps2[2] = {0, 0};
                const uint64_t sc2 = f2_pack(sl2, sl2);
#pragma unroll 1
                for (int r = 0; r < L::KT / 64; ++r) {
                    uint32_t v[64];
                    float red0, red1;
                    tmem_ld32_max(tS + r * 64, reinterpret_cast<uint32_t(&)[32]>(v[0]), red0);
                    tmem_ld32_max(tS + r * 64 + 32, reinterpret_cast<uint32_t(&)[32]>(v[32]), red1);
                    tmem_wait_ld();
                    reg_order32(reinterpret_cast<uint32_t(&)[32]>(v[0]));
                    reg_order32(reinterpret_cast<uint32_t(&)[32]>(v[32]));
                    float rm = fmaxf(red0, red1);
                    if (!full) {
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            if (r * 64 + j >= vis) v[j] = __float_as_uint(-INFINITY);
#pragma unroll
                        for (int j = 0; j < 64; j += 8)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                m4[k] = fmax3(m4[k], __uint_as_float(v[j + 2 * k]), __uint_as_float(v[j + 2 * k + 1]));
                        rm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    }
                    const float mx = rm * sl2;  // scale > 0 keeps the order; -inf stays
                    const bool up = mx > m_ref + kRescaleSlack;
                    if (__any_sync(0xffffffffu, up)) {
                        const float alpha = up ? fast_exp2(m_ref - mx) : 1.f;
                        l *= alpha;
                        ps2[0] = f2_mul(ps2[0], f2_pack(alpha, alpha));
                        ps2[1] = f2_mul(ps2[1], f2_pack(alpha, alpha));
                        a_o *= alpha;
                        any_o = true;
                        if (r > 0) {
                            a_p0 = alpha;
                            any_p0 = true;
                        }
                        if (up) m_ref = mx;
                    }
                    const float base = m_ref == -INFINITY ? 0.f : m_ref;
                    // weights, written back over S as bf16 (FP8: fp16) pairs: columns
                    // [16q, 16q+16) hold keys [32q, 32q+32), so a round only overwrites columns
                    // it has already read; the row sum adds the fp32 weights, two lanes at a time
                    const uint64_t nb2 = f2_pack(-base, -base);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(v[q * 32 + 2 * j]),
                                                               __uint_as_float(v[q * 32 + 2 * j + 1])),
                                                       sc2, nb2);
                            float x0, x1;
                            f2_unpack(x2, x0, x1);
                            const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
                            pk[j] = FP8 ? pack_f16x2(e0, e1) : pack_bf16x2(e0, e1);
                            ps2[j & 1] = f2_add(ps2[j & 1], f2_pack(e0, e1));
                        }
                        tmem_st16(tS + (2 * r + q) * 16, pk);
                    }
                }
                {
                    float a0, a1, b0, b1;
                    f2_unpack(ps2[0], a0, a1);
                    f2_unpack(ps2[1], b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                if (any_p0) {
                    // round 0's weights were taken against the reference before its move
                    tmem_wait_st();
#pragma unroll 1
                    for (int q = 0; q < 2; ++q) {
                        uint32_t w[16];
                        tmem_ld16(tS + q * 16, w);
                        tmem_wait_ld();
                        reg_order16(w);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float lo, hi;
                            if constexpr (FP8) {
                                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[j]));
                                lo = f.x;
                                hi = f.y;
                            } else {
                                lo = bf16_lo(w[j]);
                                hi = bf16_hi(w[j]);
                            }
                            w[j] = FP8 ? pack_f16x2(lo * a_p0, hi * a_p0) : pack_bf16x2(lo * a_p0, hi * a_p0);
                        }
                        tmem_st16(tS + q * 16, w);
                    }
                }
                if (any_o && ch > 0) {
                    // O holds this segment's earlier chunks (PV(c-1) is complete: the commit
                    // behind this chunk's QK covers it); rescale it.
                    const uint32_t gp = gh - 1;
                    if (!mbar_wait(&pv_done[h], gp & 1, abort_flag, a.wait_ns)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t r[32];
                        tmem_ld32(tO + q * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * a_o);
                        tmem_st32(tO + q * 32, r);
                    }
                }
                tmem_wait_st();
                if (!FP8 && h == 0 && key0 + nkeys > ctx) {
                    // The chunk runs past the context: the pool rows there may hold NaN, and
                    // 0 * NaN would poison O, so zero those V rows before PV reads them (the
                    // second half's PV is issued after the first half's, so it sees them too).
                    const uint32_t vf = 2 * gk + 1;
                    if (!mbar_wait(&kv_full[vf % NST], (vf / NST) & 1, abort_flag, a.wait_ns)) { ok = false; break; }
                    uint8_t *vst = sStage + (size_t)(vf % NST) * L::STG;
                    const int r0 = (int)(ctx - key0), nrows = nkeys - r0;
                    for (int i = tid; i < nrows * DCH * 8; i += 128) {
                        const int rr = r0 + i / (DCH * 8), rem = i % (DCH * 8);
                        *reinterpret_cast<uint4 *>(vst + (rem >> 3) * L::KV_DC + rr * 128 + ((rem & 7) << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_async_smem();
                }
                // every lane's TMEM stores are complete (wait::st); one lane arrives for the warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[h]);
            }
            if (!ok) break;
            // ---- epilogue: O / l for the tile, or the part for the merge ----
            const uint32_t gl = gh - 1;
            if (!mbar_wait(&pv_done[h], gl & 1, abort_flag, a.wait_ns)) { ok = false; break; }
            tc_fence_after();
            const bool whole = lo <= u.tile_begin && sg.end == u.tile_begin + u.tile_blocks;
            const float vsc = FP8 ? a.v_scale : 1.f;  // FP8: V elements are code x v_scale
            const float inv = vsc / l;
            const int slot = whole ? 0 : part_slot(c, u.tile_begin, T, ge);
            const int trow = tok * group + hg;  // row inside the tile
            // Staged through this warp's 32 x 128-byte buffer: each lane writes its row's
            // 128 bytes (16-byte chunks XOR-swizzled by row, so a store instruction touches
            // every bank once), then lane l reads chunk l % 8 of row 4k + l / 8 and stores it,
            // so each store instruction writes 4 whole 128-byte lines.
            uint8_t *ebuf = sEpi + (size_t)(warp - 4) * L::EPI_WARP;
            const int er = lane >> 3, ec = lane & 7;
            auto stage_and_store = [&](const uint32_t (&v)[32], auto &&dst_of_row) {
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4 *>(ebuf + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                        make_uint4(v[4 * cc], v[4 * cc + 1], v[4 * cc + 2], v[4 * cc + 3]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = 4 * k + er;  // row within the warp
                    const uint4 x = *reinterpret_cast<const uint4 *>(ebuf + rr * 128 + ((ec ^ (rr & 7)) << 4));
                    uint8_t *dst = dst_of_row(quarter * 32 + rr);
                    if (dst) *reinterpret_cast<uint4 *>(dst + ec * 16) = x;
                }
                __syncwarp();
            };
            // global address of a half row's 128-byte piece, or null for rows with no query
            auto row_ok = [&](int hr, int &tk, int &hgr) {
                tk = hr / group;
                hgr = hr - tk * group;
                return hr < half_rows && tk < half_tokens;
            };
            if (whole) {
#pragma unroll 1
                for (int hb = 0; hb < D / 64; ++hb) {  // 64 columns = 128 bytes of bf16
                    uint32_t r0[32], r1[32], v[32];
                    tmem_ld32(tO + hb * 64, r0);
                    tmem_ld32(tO + hb * 64 + 32, r1);
                    tmem_wait_ld();
                    reg_order32(r0);
                    reg_order32(r1);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        v[j] = pack_bf16x2(__uint_as_float(r0[2 * j]) * inv, __uint_as_float(r0[2 * j + 1]) * inv);
                        v[16 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]) * inv, __uint_as_float(r1[2 * j + 1]) * inv);
                    }
                    stage_and_store(v, [&](int hr) -> uint8_t * {
                        int tk, hgr;
                        if (!row_ok(hr, tk, hgr)) return nullptr;
                        const int64_t qr = u.t.q_row0 + u.qt * TPT + h * HTOK + tk;
                        return reinterpret_cast<uint8_t *>(
                                   a.out + (qr * a.num_heads + (int64_t)u.kvh * group + hgr) * D) + hb * 128;
                    });
                }
            } else {
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {  // 32 fp32 columns = 128 bytes
                    uint32_t v[32];
                    tmem_ld32(tO + q * 32, v);
                    tmem_wait_ld();
                    reg_order32(v);
                    if constexpr (FP8) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * vsc);
                    }
                    stage_and_store(v, [&](int hr) -> uint8_t * {
                        int tk, hgr;
                        if (!row_ok(hr, tk, hgr)) return nullptr;
                        const int tr = (h * HTOK + tk) * group + hgr;
                        return reinterpret_cast<uint8_t *>(a.ws_o + ((int64_t)slot * tile_rows + tr) * D) + q * 128;
                    });
                }
            }
            if (!whole && rvalid) a.ws_ml[(int64_t)slot * tile_rows + trow] = make_float2(m_ref, l);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[h]);
            f = sg.end;
        }
        if (!ok) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace pkv
