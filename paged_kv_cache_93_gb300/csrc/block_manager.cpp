// block_manager.cpp -- host-side paged KV block manager (C ABI in pkv.h).
//
// "PagedAttentionとは？KVキャッシュを分割してLLMのメモリの無駄を減らす仕組み":
//  - "PagedAttentionはブロック表で論理順序と物理配置を分ける": each sequence owns a
//    block table; it uses its current block until it is full, then appends a
//    fresh block to the table.
//  - "要求の終了で空いたブロックを再利用する具体例": blocks of a finished sequence go
//    back to the pool and can serve any other sequence; nothing is compacted.
//  - "共通ブロックの共有とコピーオンライト": several tables may point at one physical
//    block; a reference count keeps it alive while any sequence uses it, and a
//    write into a shared, partly filled last block first duplicates it.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

struct pkv_block_manager {
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
    };
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> free_list;   // back() is handed out next
    std::vector<int32_t> refs;
    std::unordered_map<int64_t, Seq> seqs;
    int64_t next_id = 0;

    int32_t take() {
        int32_t b = free_list.back();
        free_list.pop_back();
        refs[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--refs[b] == 0) free_list.push_back(b);
    }
};

extern "C" pkv_block_manager *pkv_bm_create(int32_t num_blocks, int32_t block_size,
                                            const int32_t *initial_order) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    auto *bm = new (std::nothrow) pkv_block_manager;
    if (!bm) return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refs.assign(num_blocks, 0);
    bm->free_list.resize(num_blocks);
    if (initial_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            const int32_t b = initial_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete bm;
                return nullptr;
            }
            seen[b] = 1;
        }
    }
    // Free list is a stack: the first block to hand out goes last.
    for (int32_t i = 0; i < num_blocks; ++i)
        bm->free_list[num_blocks - 1 - i] = initial_order ? initial_order[i] : i;
    return bm;
}

extern "C" void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

extern "C" int pkv_bm_add_sequence(pkv_block_manager *bm, int64_t *seq_id) {
    if (!bm || !seq_id) return PKV_ERR_INVALID_ARG;
    const int64_t id = bm->next_id++;
    bm->seqs.emplace(id, pkv_block_manager::Seq{});
    *seq_id = id;
    return PKV_OK;
}

extern "C" int pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t *child) {
    if (!bm || !child) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end()) return PKV_ERR_NOT_FOUND;
    pkv_block_manager::Seq copy = it->second;
    for (int32_t b : copy.table) ++bm->refs[b];
    const int64_t id = bm->next_id++;
    bm->seqs.emplace(id, std::move(copy));
    *child = id;
    return PKV_OK;
}

extern "C" int pkv_bm_append(pkv_block_manager *bm, int64_t seq, int32_t num_tokens,
                             int64_t *slots_out, int32_t *cow_src, int32_t *cow_dst,
                             int32_t cow_capacity, int32_t *num_cow) {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !slots_out) || !num_cow)
        return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_NOT_FOUND;
    pkv_block_manager::Seq &s = it->second;
    *num_cow = 0;
    if (num_tokens == 0) return PKV_OK;
    const int64_t bs = bm->block_size;
    const int64_t used_in_last = s.len % bs;            // tokens already in a partial last block
    const bool has_partial = used_in_last != 0;
    const bool cow = has_partial && bm->refs[s.table.back()] > 1;
    const int64_t new_len = s.len + num_tokens;
    const int64_t blocks_after = (new_len + bs - 1) / bs;
    const int64_t fresh = blocks_after - int64_t(s.table.size()) + (cow ? 1 : 0);
    if (cow && (!cow_src || !cow_dst || cow_capacity < 1)) return PKV_ERR_INVALID_ARG;
    if (fresh > int64_t(bm->free_list.size())) return PKV_ERR_NO_SPACE;

    if (cow) {
        const int32_t old_block = s.table.back();
        const int32_t copy = bm->take();
        bm->release(old_block);     // still referenced by the other sequences
        s.table.back() = copy;
        cow_src[0] = old_block;
        cow_dst[0] = copy;
        *num_cow = 1;
    }
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int64_t pos = s.len + t;
        if (pos / bs >= int64_t(s.table.size())) s.table.push_back(bm->take());
        slots_out[t] = int64_t(s.table[pos / bs]) * bs + pos % bs;
    }
    s.len = new_len;
    return PKV_OK;
}

extern "C" int pkv_bm_free(pkv_block_manager *bm, int64_t seq) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_NOT_FOUND;
    // Release in reverse so the sequence's first block is the next one reused.
    for (auto b = it->second.table.rbegin(); b != it->second.table.rend(); ++b) bm->release(*b);
    bm->seqs.erase(it);
    return PKV_OK;
}

extern "C" int pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq, int32_t *table_out,
                                  int32_t capacity, int32_t *num_blocks, int64_t *seq_len) {
    if (!bm || capacity < 0) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_NOT_FOUND;
    const auto &t = it->second.table;
    if (num_blocks) *num_blocks = int32_t(t.size());
    if (seq_len) *seq_len = it->second.len;
    if (int64_t(t.size()) > capacity) return PKV_ERR_SHAPE;
    if (table_out && !t.empty()) std::memcpy(table_out, t.data(), t.size() * sizeof(int32_t));
    return PKV_OK;
}

extern "C" int32_t pkv_bm_num_free(const pkv_block_manager *bm) {
    return bm ? int32_t(bm->free_list.size()) : -1;
}

extern "C" int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->refs[block];
}
