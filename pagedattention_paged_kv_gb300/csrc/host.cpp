// host.cpp -- host-side parts of libpagedkv: slot mapping and the block manager.
//
// "Servis Motor İçleri: PagedAttention, Sürekli Batching, parçalanmış Prefill"
// (aiengineeringfromscratch.com, Phase 17 - 04), "PagedAttention as a virtual memory
// system": a sequence's KV lives in fixed-size blocks, its block table maps logical
// token positions to physical block ids, a growing sequence takes one more block and a
// finished one returns its blocks to the pool.
// "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn) §2.2 BlockManager:
// allocate(n) hands out the first n ids of the free list or raises out-of-memory;
// free(ids) appends them back.
#include <algorithm>
#include <cstdint>
#include <deque>
#include <new>
#include <vector>

#include "../../include/pagedkv.h"

extern "C" int pkv_slot_mapping(int64_t *host_slot_mapping, const int32_t *host_block_tables,
                                int max_blocks_per_seq, const int32_t *host_token_seq,
                                const int32_t *host_token_pos, int64_t num_tokens,
                                int block_size) {
    if (num_tokens < 0 || block_size <= 0 || max_blocks_per_seq < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!host_slot_mapping || !host_block_tables || !host_token_seq || !host_token_pos)
        return PKV_ERR_INVALID_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int32_t seq = host_token_seq[t];
        if (seq < 0) {
            host_slot_mapping[t] = -1;
            continue;
        }
        const int32_t pos = host_token_pos[t];
        if (pos < 0) return PKV_ERR_INVALID_ARG;
        const int64_t logical = pos / block_size;
        if (logical >= max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
        const int32_t physical = host_block_tables[(int64_t)seq * max_blocks_per_seq + logical];
        if (physical < 0) return PKV_ERR_INVALID_ARG;
        host_slot_mapping[t] = (int64_t)physical * block_size + pos % block_size;
    }
    return PKV_OK;
}

// Blocks carry a reference count so that several sequences can hold the same block
// read-only: "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn) §4.3 -- requests
// sharing a system-prompt prefix reuse one set of read-only blocks.  A block returns to
// the free list when its last holder frees it.
struct pkv_block_manager {
    int64_t num_blocks;
    int block_size;
    std::deque<int32_t> free_list;  // head = next to hand out
    std::vector<int32_t> refs;      // holders of each block (0 = free)
};

extern "C" pkv_block_manager *pkv_block_manager_create(int64_t num_blocks, int block_size) {
    if (num_blocks < 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
    auto *bm = new (std::nothrow) pkv_block_manager;
    if (!bm) return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refs.assign((size_t)num_blocks, 0);
    for (int64_t b = 0; b < num_blocks; ++b) bm->free_list.push_back((int32_t)b);
    return bm;
}

extern "C" void pkv_block_manager_destroy(pkv_block_manager *bm) { delete bm; }

extern "C" int pkv_block_manager_allocate(pkv_block_manager *bm, int64_t n, int32_t *host_ids_out) {
    if (!bm || n < 0 || (n > 0 && !host_ids_out)) return PKV_ERR_INVALID_ARG;
    if ((int64_t)bm->free_list.size() < n) return PKV_ERR_OOM;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = bm->free_list.front();
        bm->free_list.pop_front();
        bm->refs[(size_t)b] = 1;
        host_ids_out[i] = b;
    }
    return PKV_OK;
}

// Counts how often each id occurs in host_ids; false if an id is outside the pool or
// (need_held) occurs more often than it is held.
static bool count_ids(const pkv_block_manager *bm, const int32_t *host_ids, int64_t n, bool need_held,
                      std::vector<std::pair<int32_t, int32_t>> &counts) {
    std::vector<int32_t> ids(host_ids, host_ids + n);
    std::sort(ids.begin(), ids.end());
    for (int64_t i = 0; i < n;) {
        const int32_t b = ids[(size_t)i];
        if (b < 0 || b >= bm->num_blocks) return false;
        int64_t j = i;
        while (j < n && ids[(size_t)j] == b) ++j;
        const int32_t c = (int32_t)(j - i);
        if (bm->refs[(size_t)b] == 0 || (need_held && c > bm->refs[(size_t)b])) return false;
        counts.emplace_back(b, c);
        i = j;
    }
    return true;
}

extern "C" int pkv_block_manager_free(pkv_block_manager *bm, const int32_t *host_ids, int64_t n) {
    if (!bm || n < 0 || (n > 0 && !host_ids)) return PKV_ERR_INVALID_ARG;
    // Validate everything first so that a bad call changes nothing.
    std::vector<std::pair<int32_t, int32_t>> counts;
    if (!count_ids(bm, host_ids, n, true, counts)) return PKV_ERR_INVALID_ARG;
    // Blocks whose last holder leaves go back in the order the caller listed them.
    for (auto &bc : counts) bm->refs[(size_t)bc.first] -= bc.second;
    std::vector<uint8_t> queued;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = host_ids[i];
        if (bm->refs[(size_t)b] == 0) {
            bm->refs[(size_t)b] = -1;  // mark as queued (restored to 0 below)
            bm->free_list.push_back(b);
        }
    }
    for (auto &bc : counts)
        if (bm->refs[(size_t)bc.first] < 0) bm->refs[(size_t)bc.first] = 0;
    return PKV_OK;
}

extern "C" int64_t pkv_block_manager_num_free(const pkv_block_manager *bm) {
    return bm ? (int64_t)bm->free_list.size() : -1;
}

extern "C" int pkv_block_manager_share(pkv_block_manager *bm, const int32_t *host_ids, int64_t n) {
    if (!bm || n < 0 || (n > 0 && !host_ids)) return PKV_ERR_INVALID_ARG;
    std::vector<std::pair<int32_t, int32_t>> counts;
    if (!count_ids(bm, host_ids, n, false, counts)) return PKV_ERR_INVALID_ARG;
    for (auto &bc : counts) bm->refs[(size_t)bc.first] += bc.second;
    return PKV_OK;
}

extern "C" int pkv_block_manager_ref_count(const pkv_block_manager *bm, int32_t id) {
    if (!bm || id < 0 || id >= bm->num_blocks) return PKV_ERR_INVALID_ARG;
    return bm->refs[(size_t)id];
}

extern "C" int pkv_block_manager_copy_on_write(pkv_block_manager *bm, int32_t id, int32_t *host_new_id) {
    if (!bm || !host_new_id || id < 0 || id >= bm->num_blocks || bm->refs[(size_t)id] == 0)
        return PKV_ERR_INVALID_ARG;
    if (bm->refs[(size_t)id] == 1) {  // sole holder: write in place
        *host_new_id = id;
        return 0;
    }
    if (bm->free_list.empty()) return PKV_ERR_OOM;
    const int32_t nb = bm->free_list.front();
    bm->free_list.pop_front();
    bm->refs[(size_t)nb] = 1;
    bm->refs[(size_t)id] -= 1;
    *host_new_id = nb;
    return 1;
}
