// paged_prefill.cu -- chunked-prefill attention over a block-paged KV cache (sm_103a).
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
//  * A tile is 16 query tokens x the `group` query heads of one KV head (128 rows for
//    Llama-70B shapes): one K/V block read from shared memory feeds 128 query rows,
//    enough reuse for the work to be tensor-bound.  Eight consumer warps each own 16
//    rows and run S = Q K^T and O += P V as m16n8k16 bf16 MMAs with fp32 accumulation
//    and an fp32 online softmax; the S fragments become the P operand directly.
//  * The units are (tile, 16-token key block) pairs; causal tiles stop at the block
//    holding their last query's position.  A persistent grid (one CTA per SM) takes
//    equal contiguous shares of the flat unit list, so long prefixes split across
//    CTAs and no SM idles in a tail; split tiles are merged by log-sum-exp weights.
//  * A producer warp streams each key block (K, then V, of one KV head: 16 rows x
//    head_dim) with TMA into a ring of 128-byte-swizzled shared-memory stages.
//  * Waits are bounded in time; no CTA waits on another CTA.
#include "attn_block.cuh"
#include "merge.cuh"
#include "paged_prefill.cuh"
#include "pkv_split.cuh"

namespace pkv {

namespace {

constexpr int kBS = 16;

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
__device__ void build_seq_prefix(const PrefillArgs &a, int64_t *pre, int64_t *scan_tmp) {
    const int S = a.num_seqs;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (S + nt - 1) / nt;
    const int beg = min(S, tid * per), end = min(S, beg + per);
    int64_t local = 0;
    for (int s = beg; s < end; ++s) local += seq_units(a, s, blockIdx.x == 0);
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

template <int D>
__global__ void __launch_bounds__(288, 1)
paged_prefill_kernel(const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap v_map, const PrefillArgs a) {
    constexpr int KSTEPS = D / 16;
    constexpr int NT_D = D / 8;
    constexpr int DCH = D / 64;
    constexpr uint32_t kStageBytes = kBS * D * 2;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NST = a.num_stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NST * kStageBytes);
    uint64_t *empty = full + NST;
    int64_t *scan_tmp = reinterpret_cast<int64_t *>(empty + NST);  // 32 entries
    volatile int *abort_flag = reinterpret_cast<int *>(scan_tmp + 32);
    int64_t *pre = scan_tmp + 34;

    const int group = a.group, TPT = a.tokens_per_tile;
    const int rows = TPT * group;
    const int ncw = (rows + 15) / 16;
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
    pdl_wait();
    pdl_trigger();
    build_seq_prefix(a, pre, scan_tmp);
    const int64_t T = pre[a.num_seqs];
    const int ge = split_ctas(T, a.grid, 4);
    if (blockIdx.x == 0) write_jobs_and_invalid_rows<D>(a, pre, T, ge);
    if ((int)blockIdx.x >= ge || T == 0) return;
    const int c = blockIdx.x;
    const int64_t lo = share_begin(c, T, ge), hi = share_begin(c + 1, T, ge);

    if (warp == ncw) {
        // ------------------------------ producer ------------------------------
        const uint64_t policy = l2_policy_evict_normal();
        uint32_t stage = 0, phase = 0, issued = 0;
        bool ok = true;
        for (int64_t f0 = lo; f0 < hi && ok; f0 += 32) {
            const int64_t f = f0 + lane;
            int bid = -1, kvh = 0;
            if (f < hi) {
                UnitPos u;
                locate(a, pre, f, u);
                kvh = u.kvh;
                bid = a.block_tables[(int64_t)u.s * a.max_blocks_per_seq + u.kb];
                if (bid < 0 || (int64_t)bid >= a.num_blocks) {
                    flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                    bid = -1;
                }
            }
            const int n = (int)min64(32, hi - f0);
            for (int j = 0; j < n; ++j) {
                const int b = __shfl_sync(0xffffffffu, bid, j);
                const int h = __shfl_sync(0xffffffffu, kvh, j);
                if (lane == 0) {
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[stage], kStageBytes);
                        uint8_t *dst = smem + (size_t)stage * kStageBytes;
                        const CUtensorMap *map = kv == 0 ? &k_map : &v_map;
#pragma unroll
                        for (int dc = 0; dc < DCH; ++dc)
                            tma_load_5d(dst + dc * (kBS * 128), map, &full[stage], 0, 0, h, dc,
                                        b, policy);
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
    const int g_row = lane >> 2, q4 = lane & 3;
    const int ra = warp * 16 + g_row, rb = ra + 8;  // this lane's two tile rows
    const uint32_t smem_base = smem_u32(smem);
    const float sl2 = a.scale_log2;
    uint32_t stage = 0, phase = 0;
    int64_t f = lo;
    RowState<D> st;
    while (f < hi) {
        UnitPos u;
        locate(a, pre, f, u);
        const int64_t tile_end = u.tile_begin + u.tile_blocks;
        const int64_t seg_end = min64(hi, tile_end);
        const int tile_tokens = (int)min64(TPT, u.t.q_len - u.qt * TPT);
        const int tok_a = ra / group, tok_b = rb / group;
        const bool va = ra < rows && tok_a < tile_tokens;
        const bool vb = rb < rows && tok_b < tile_tokens;
        const int64_t first_pos = (int64_t)(u.t.ctx - u.t.q_len) + u.qt * TPT;
        const int ctx = u.t.ctx;
        // keys a row may see: [0, lim)
        const int64_t lim_a = a.causal ? min64(first_pos + min(tok_a, tile_tokens - 1) + 1, ctx) : ctx;
        const int64_t lim_b = a.causal ? min64(first_pos + min(tok_b, tile_tokens - 1) + 1, ctx) : ctx;
        // keys every row of the warp may see (for the no-mask fast path)
        const int64_t lim_warp = a.causal
            ? min64(first_pos + min((warp * 16) / group, tile_tokens - 1) + 1, ctx) : ctx;

        uint32_t qa[KSTEPS][4];
        {
            const int64_t qrow_a = u.t.q_row0 + u.qt * TPT + tok_a;
            const int64_t qrow_b = u.t.q_row0 + u.qt * TPT + tok_b;
            const uint32_t *pa = reinterpret_cast<const uint32_t *>(
                a.q + (qrow_a * a.num_heads + (int64_t)u.kvh * group + ra % group) * D);
            const uint32_t *pb = reinterpret_cast<const uint32_t *>(
                a.q + (qrow_b * a.num_heads + (int64_t)u.kvh * group + rb % group) * D);
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const int col = ks * 16 + 2 * q4;
                qa[ks][0] = va ? __ldg(pa + col / 2) : 0u;
                qa[ks][1] = vb ? __ldg(pb + col / 2) : 0u;
                qa[ks][2] = va ? __ldg(pa + (col + 8) / 2) : 0u;
                qa[ks][3] = vb ? __ldg(pb + (col + 8) / 2) : 0u;
            }
        }
        st.reset();

        bool ok = true;
        for (; f < seg_end; ++f) {
            const int64_t key0 = (f - u.tile_begin) * kBS;
            if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
            float sacc[2][4];
            qk_block<D>(sacc, qa, smem_base + stage * kStageBytes, kBS * 128, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1; }

            if (key0 + kBS <= lim_warp) {  // the whole block is visible to every row
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    sacc[0][i] *= sl2;
                    sacc[1][i] *= sl2;
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int64_t key = key0 + nt * 8 + 2 * q4 + e;
                        sacc[nt][e] = key < lim_a ? sacc[nt][e] * sl2 : -INFINITY;
                        sacc[nt][2 + e] = key < lim_b ? sacc[nt][2 + e] * sl2 : -INFINITY;
                    }
            }
            uint32_t pa[4];
            softmax_update<D>(st, sacc, pa);

            if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
            if (key0 + kBS <= ctx)
                pv_block<D, false>(st, pa, smem_base + stage * kStageBytes, kBS * 128, kBS, lane);
            else
                pv_block<D, true>(st, pa, smem_base + stage * kStageBytes, kBS * 128,
                                  (int)(ctx - key0), lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1; }
        }
        if (!ok) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
            return;
        }

        finish_sums<D>(st);
        const bool whole = lo <= u.tile_begin && seg_end == tile_end;
        if (whole) {
            const float inv0 = 1.f / st.l0, inv1 = 1.f / st.l1;
            const int64_t qrow_a = u.t.q_row0 + u.qt * TPT + tok_a;
            const int64_t qrow_b = u.t.q_row0 + u.qt * TPT + tok_b;
            __nv_bfloat16 *oa = a.out + (qrow_a * a.num_heads + (int64_t)u.kvh * group + ra % group) * D;
            __nv_bfloat16 *ob = a.out + (qrow_b * a.num_heads + (int64_t)u.kvh * group + rb % group) * D;
#pragma unroll
            for (int n = 0; n < NT_D; ++n) {
                const int col = n * 8 + 2 * q4;
                if (va) *reinterpret_cast<uint32_t *>(oa + col) = pack_bf16x2(st.o[n][0] * inv0, st.o[n][1] * inv0);
                if (vb) *reinterpret_cast<uint32_t *>(ob + col) = pack_bf16x2(st.o[n][2] * inv1, st.o[n][3] * inv1);
            }
        } else {
            const int slot = part_slot(c, u.tile_begin, T, ge);
            float *ws = a.ws_o + (int64_t)slot * rows * D;
            float2 *ml = a.ws_ml + (int64_t)slot * rows;
#pragma unroll
            for (int n = 0; n < NT_D; ++n) {
                const int col = n * 8 + 2 * q4;
                if (va) *reinterpret_cast<float2 *>(ws + (int64_t)ra * D + col) = make_float2(st.o[n][0], st.o[n][1]);
                if (vb) *reinterpret_cast<float2 *>(ws + (int64_t)rb * D + col) = make_float2(st.o[n][2], st.o[n][3]);
            }
            if (q4 == 0) {
                if (va) ml[ra] = make_float2(st.m0, st.l0);
                if (vb) ml[rb] = make_float2(st.m1, st.l1);
            }
        }
        f = seg_end;
    }
}

// ---- host side -------------------------------------------------------------------

int plan_prefill(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int sms,
                 int smem_optin, PrefillPlan *p) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads) return PKV_ERR_UNSUPPORTED;
    p->group = num_heads / num_kv_heads;
    if (p->group > 8) return PKV_ERR_UNSUPPORTED;
    p->tokens_per_tile = 16 * (8 / p->group);
    p->rows = p->tokens_per_tile * p->group;
    p->warps = (p->rows + 15) / 16;
    p->grid = sms < 256 ? sms : 256;  // the merge kernel holds <= 256 parts per tile
    p->max_seqs = num_seqs;
    p->stage_bytes = kBS * head_dim * 2;
    const size_t fixed = 1024 + 34 * 8 + 8 * (size_t)(num_seqs + 1) + 8;
    int nst = (int)(((int64_t)smem_optin - (int64_t)fixed) / (p->stage_bytes + 16));
    if (nst > 32) nst = 32;
    if (nst < 4) return PKV_ERR_UNSUPPORTED;
    p->num_stages = nst;
    p->smem = fixed + (size_t)nst * (p->stage_bytes + 16);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    p->off_jobs = 0;
    p->off_ml = up(sizeof(MergeJob) * (size_t)p->grid);
    p->off_o = p->off_ml + up(2 * (size_t)p->grid * p->rows * 8);
    p->ws_bytes = p->off_o + up(2 * (size_t)p->grid * p->rows * head_dim * 4);
    return PKV_OK;
}

template <int D>
static cudaError_t launch_prefill_d(const CUtensorMap &k_map, const CUtensorMap &v_map,
                                    const PrefillArgs &a, const PrefillPlan &p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(paged_prefill_kernel<D>, dim3(a.grid), dim3((p.warps + 1) * 32), p.smem, stream,
                   k_map, v_map, a);
    if (e != cudaSuccess) return e;
    MergeArgs m;
    m.jobs = a.ws_jobs;
    m.ws_ml = a.ws_ml;
    m.ws_o = a.ws_o;
    m.out = a.out;
    m.slot_rows = p.rows;
    m.num_heads = a.num_heads;
    return launch_merge<D>(m, a.grid, stream);
}

cudaError_t launch_paged_prefill(int head_dim, const CUtensorMap &k_map, const CUtensorMap &v_map,
                                 const PrefillArgs &a, const PrefillPlan &p, cudaStream_t stream) {
    return head_dim == 128 ? launch_prefill_d<128>(k_map, v_map, a, p, stream)
                           : launch_prefill_d<64>(k_map, v_map, a, p, stream);
}

}  // namespace pkv
