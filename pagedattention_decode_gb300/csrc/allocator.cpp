// allocator.cpp -- host block allocator and per-sequence block tables (a1, a9).
//
// "nanoserve day 14: the block allocator", section "What I learned": free ids
// on a stack, handed-out ids tracked separately so that every id is in exactly
// one of the two; a double free is a loud error; allocate_for(n) takes
// ceil(n / block_size) blocks or none.  Here the handed-out set is the set of
// ids with refcount > 0 (one int per id, O(1) membership).
//
// "How to Implement Paged Attention in PyTorch and vLLM", section "Build the
// block allocator and block tables in PyTorch": the stack starts as ids
// num_blocks-1 .. 0, a sequence takes a new block when pos % block_size == 0,
// the token's slot is table[pos / block_size] * block_size + pos % block_size,
// and freeing a sequence pushes its ids in table order.
//
// "Build a paged KV cache manager from scratch", Steps 2-3 and the
// copy-on-write paragraph: refcounts (1 on allocation, +1 per share/fork),
// forks share every id, a shared block is copied on the first divergent write.
#include <algorithm>
#include <map>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "internal.h"

struct pkv_allocator {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> free_stack;  // top = back()
    std::vector<int32_t> refcount;    // 0 = on the free stack
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
        bool live = true;
    };
    std::vector<Seq> seqs;
    pkv_alloc_counters counters{0, 0, 0, 0};
    mutable std::mutex mu;

    // Prefix trie ("Build a paged KV cache manager from scratch", Step 4):
    // children keyed by one whole block of token ids; each node holds one
    // reference to its block.  Node 0 is the root.
    struct Node {
        std::map<std::vector<int32_t>, int32_t> children;
        int32_t parent = -1;
        std::vector<int32_t> key;
        int32_t block = -1;
        int64_t last_used = 0;
        bool live = true;
    };
    std::vector<Node> nodes{Node{}};
    int64_t clock = 0;
    int32_t trie_nodes = 0;

    int32_t used() const { return num_blocks - (int32_t)free_stack.size(); }

    int32_t pop() {
        int32_t id = free_stack.back();
        free_stack.pop_back();
        refcount[id] = 1;
        counters.allocs += 1;
        counters.peak_used = std::max<int64_t>(counters.peak_used, used());
        return id;
    }

    void release_one(int32_t id) {  // caller checked refcount[id] > 0
        if (--refcount[id] == 0) {
            free_stack.push_back(id);
            counters.frees += 1;
        }
    }

    bool valid_id(int32_t id) const { return id >= 0 && id < num_blocks; }
    bool live_seq(int32_t s) const { return s >= 0 && s < (int32_t)seqs.size() && seqs[s].live; }
};

using Guard = std::lock_guard<std::mutex>;

extern "C" {

pkv_status pkv_alloc_create(int32_t num_blocks, int32_t block_size, pkv_allocator **out) {
    PKV_CHECK_ARG(out, PKV_ERR_INVALID_ARG, "out is NULL");
    PKV_CHECK_ARG(num_blocks > 0 && block_size > 0, PKV_ERR_INVALID_ARG,
                  "num_blocks (%d) and block_size (%d) must be positive", num_blocks, block_size);
    auto *a = new pkv_allocator();
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->free_stack.resize(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) a->free_stack[i] = num_blocks - 1 - i;
    a->refcount.assign(num_blocks, 0);
    *out = a;
    return pkv::ok();
}

void pkv_alloc_destroy(pkv_allocator *a) { delete a; }

pkv_status pkv_alloc_set_free_order(pkv_allocator *a, const int32_t *order, int32_t n) {
    PKV_CHECK_ARG(a && (order || n == 0), PKV_ERR_INVALID_ARG, "NULL argument");
    Guard g(a->mu);
    PKV_CHECK_ARG(n == (int32_t)a->free_stack.size(), PKV_ERR_SHAPE,
                  "order has %d ids, %zu are free", n, a->free_stack.size());
    std::vector<char> seen(a->num_blocks, 0);
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = order[i];
        PKV_CHECK_ARG(a->valid_id(id) && a->refcount[id] == 0 && !seen[id], PKV_ERR_OUT_OF_RANGE,
                      "order[%d] = %d is not a free id (or repeats)", i, id);
        seen[id] = 1;
    }
    for (int32_t i = 0; i < n; ++i) a->free_stack[i] = order[n - 1 - i];
    return pkv::ok();
}

pkv_status pkv_alloc_allocate(pkv_allocator *a, int32_t *block_id) {
    PKV_CHECK_ARG(a && block_id, PKV_ERR_INVALID_ARG, "NULL argument");
    Guard g(a->mu);
    PKV_CHECK_ARG(!a->free_stack.empty(), PKV_ERR_EXHAUSTED, "all %d blocks allocated", a->num_blocks);
    *block_id = a->pop();
    return pkv::ok();
}

int64_t pkv_alloc_blocks_needed(const pkv_allocator *a, int64_t num_tokens) {
    if (!a || num_tokens < 0) return -1;
    return (num_tokens + a->block_size - 1) / a->block_size;
}

pkv_status pkv_alloc_allocate_for(pkv_allocator *a, int64_t num_tokens, int32_t *out_ids,
                                  int32_t capacity, int32_t *num_out) {
    PKV_CHECK_ARG(a && num_out && (out_ids || capacity == 0), PKV_ERR_INVALID_ARG, "NULL argument");
    PKV_CHECK_ARG(num_tokens >= 0, PKV_ERR_INVALID_ARG, "negative token count");
    Guard g(a->mu);
    int64_t need = (num_tokens + a->block_size - 1) / a->block_size;
    PKV_CHECK_ARG(need <= capacity, PKV_ERR_INVALID_ARG, "capacity %d < %lld blocks", capacity,
                  (long long)need);
    PKV_CHECK_ARG(need <= (int64_t)a->free_stack.size(), PKV_ERR_EXHAUSTED,
                  "need %lld blocks, %zu free", (long long)need, a->free_stack.size());
    for (int64_t i = 0; i < need; ++i) out_ids[i] = a->pop();
    *num_out = (int32_t)need;
    return pkv::ok();
}

pkv_status pkv_alloc_free(pkv_allocator *a, int32_t id) {
    PKV_CHECK_ARG(a, PKV_ERR_INVALID_ARG, "NULL allocator");
    Guard g(a->mu);
    PKV_CHECK_ARG(a->valid_id(id) && a->refcount[id] > 0, PKV_ERR_DOUBLE_FREE,
                  "block %d is not handed out", id);
    a->release_one(id);
    return pkv::ok();
}

pkv_status pkv_alloc_free_all(pkv_allocator *a, const int32_t *ids, int32_t n) {
    PKV_CHECK_ARG(a && (ids || n == 0) && n >= 0, PKV_ERR_INVALID_ARG, "bad argument");
    Guard g(a->mu);
    std::unordered_map<int32_t, int32_t> count;
    for (int32_t i = 0; i < n; ++i) {
        PKV_CHECK_ARG(a->valid_id(ids[i]), PKV_ERR_DOUBLE_FREE, "block %d is not in the pool", ids[i]);
        count[ids[i]] += 1;
    }
    for (auto &kv : count)
        PKV_CHECK_ARG(a->refcount[kv.first] >= kv.second, PKV_ERR_DOUBLE_FREE,
                      "block %d freed %d times, held %d", kv.first, kv.second, a->refcount[kv.first]);
    for (int32_t i = 0; i < n; ++i) a->release_one(ids[i]);
    return pkv::ok();
}

pkv_status pkv_alloc_retain(pkv_allocator *a, int32_t id) {
    PKV_CHECK_ARG(a, PKV_ERR_INVALID_ARG, "NULL allocator");
    Guard g(a->mu);
    PKV_CHECK_ARG(a->valid_id(id) && a->refcount[id] > 0, PKV_ERR_DOUBLE_FREE,
                  "block %d is not handed out", id);
    a->refcount[id] += 1;
    return pkv::ok();
}

int32_t pkv_alloc_refcount(const pkv_allocator *a, int32_t id) {
    if (!a) return -1;
    Guard g(a->mu);
    return a->valid_id(id) ? a->refcount[id] : -1;
}

int32_t pkv_alloc_num_free(const pkv_allocator *a) {
    if (!a) return -1;
    Guard g(a->mu);
    return (int32_t)a->free_stack.size();
}

pkv_status pkv_alloc_counters_get(const pkv_allocator *a, pkv_alloc_counters *out) {
    PKV_CHECK_ARG(a && out, PKV_ERR_INVALID_ARG, "NULL argument");
    Guard g(a->mu);
    *out = a->counters;
    return pkv::ok();
}

// ---- sequences ---------------------------------------------------------------

pkv_status pkv_seq_create(pkv_allocator *a, const int32_t *shared_ids, int32_t n_shared,
                          int64_t shared_tokens, int32_t *seq_id) {
    PKV_CHECK_ARG(a && seq_id && n_shared >= 0 && (shared_ids || n_shared == 0),
                  PKV_ERR_INVALID_ARG, "bad argument");
    Guard g(a->mu);
    PKV_CHECK_ARG(shared_tokens == (int64_t)n_shared * a->block_size, PKV_ERR_SHAPE,
                  "only whole blocks are shared: %lld tokens for %d blocks of %d",
                  (long long)shared_tokens, n_shared, a->block_size);
    for (int32_t i = 0; i < n_shared; ++i)
        PKV_CHECK_ARG(a->valid_id(shared_ids[i]) && a->refcount[shared_ids[i]] > 0,
                      PKV_ERR_DOUBLE_FREE, "shared block %d is not handed out", shared_ids[i]);
    pkv_allocator::Seq s;
    s.table.assign(shared_ids, shared_ids + n_shared);
    s.len = shared_tokens;
    for (int32_t id : s.table) a->refcount[id] += 1;
    a->seqs.push_back(std::move(s));
    *seq_id = (int32_t)a->seqs.size() - 1;
    return pkv::ok();
}

pkv_status pkv_seq_fork(pkv_allocator *a, int32_t seq_id, int32_t *child_id) {
    PKV_CHECK_ARG(a && child_id, PKV_ERR_INVALID_ARG, "NULL argument");
    Guard g(a->mu);
    PKV_CHECK_ARG(a->live_seq(seq_id), PKV_ERR_OUT_OF_RANGE, "sequence %d is not live", seq_id);
    pkv_allocator::Seq c;
    c.table = a->seqs[seq_id].table;
    c.len = a->seqs[seq_id].len;
    for (int32_t id : c.table) a->refcount[id] += 1;
    a->seqs.push_back(std::move(c));
    *child_id = (int32_t)a->seqs.size() - 1;
    return pkv::ok();
}

pkv_status pkv_seq_free(pkv_allocator *a, int32_t seq_id) {
    PKV_CHECK_ARG(a, PKV_ERR_INVALID_ARG, "NULL allocator");
    Guard g(a->mu);
    PKV_CHECK_ARG(seq_id >= 0 && seq_id < (int32_t)a->seqs.size(), PKV_ERR_OUT_OF_RANGE,
                  "unknown sequence %d", seq_id);
    auto &s = a->seqs[seq_id];
    if (!s.live) return pkv::ok();  // freeing a finished sequence again is harmless
    for (int32_t id : s.table) a->release_one(id);
    s.table.clear();
    s.table.shrink_to_fit();
    s.len = 0;
    s.live = false;
    return pkv::ok();
}

pkv_status pkv_seq_append(pkv_allocator *a, const int32_t *seq_ids, const int32_t *counts, int32_t n,
                          int64_t *out_slots, int64_t slot_capacity, int64_t *out_pairs,
                          int32_t pair_capacity, int32_t *num_pairs) {
    PKV_CHECK_ARG(a && num_pairs && n >= 0 && (seq_ids || n == 0), PKV_ERR_INVALID_ARG, "bad argument");
    Guard g(a->mu);
    const int32_t bs = a->block_size;
    // validate and count what the call needs before anything moves
    int64_t total_tokens = 0, need_blocks = 0, need_pairs = 0;
    std::unordered_map<int32_t, int32_t> seen, tail_delta;
    for (int32_t i = 0; i < n; ++i) {
        int32_t sid = seq_ids[i];
        PKV_CHECK_ARG(a->live_seq(sid), PKV_ERR_OUT_OF_RANGE, "sequence %d is not live", sid);
        PKV_CHECK_ARG(seen[sid]++ == 0, PKV_ERR_INVALID_ARG, "sequence %d appears twice", sid);
        int32_t cnt = counts ? counts[i] : 1;
        PKV_CHECK_ARG(cnt >= 0, PKV_ERR_INVALID_ARG, "negative count for sequence %d", sid);
        const auto &s = a->seqs[sid];
        total_tokens += cnt;
        if (cnt == 0) continue;
        int64_t pos = s.len;
        if (pos % bs != 0) {
            int32_t tail = s.table[pos / bs];
            int32_t rc = a->refcount[tail] + tail_delta[tail];
            if (rc > 1) {
                need_blocks += 1;
                need_pairs += 1;
                tail_delta[tail] -= 1;
            }
        }
        // new blocks opened by positions pos .. pos+cnt-1 that are multiples of bs
        int64_t first = (pos + bs - 1) / bs, last = (pos + cnt - 1) / bs;
        if (last >= first) need_blocks += last - first + 1;
    }
    PKV_CHECK_ARG(total_tokens <= slot_capacity && (out_slots || total_tokens == 0), PKV_ERR_INVALID_ARG,
                  "slot capacity %lld < %lld tokens", (long long)slot_capacity, (long long)total_tokens);
    PKV_CHECK_ARG(need_pairs <= pair_capacity && (out_pairs || need_pairs == 0), PKV_ERR_INVALID_ARG,
                  "pair capacity %d < %lld", pair_capacity, (long long)need_pairs);
    PKV_CHECK_ARG(need_blocks <= (int64_t)a->free_stack.size(), PKV_ERR_EXHAUSTED,
                  "need %lld blocks, %zu free", (long long)need_blocks, a->free_stack.size());
    int64_t k = 0;
    int32_t np = 0;
    for (int32_t i = 0; i < n; ++i) {
        auto &s = a->seqs[seq_ids[i]];
        int32_t cnt = counts ? counts[i] : 1;
        for (int32_t j = 0; j < cnt; ++j) {
            int64_t pos = s.len;
            int64_t off = pos % bs;
            if (off == 0) {
                s.table.push_back(a->pop());
            } else {
                int32_t &tail = s.table[pos / bs];
                if (a->refcount[tail] > 1) {
                    int32_t dst = a->pop();
                    out_pairs[2 * np] = tail;
                    out_pairs[2 * np + 1] = dst;
                    ++np;
                    a->counters.cow_copies += 1;
                    a->release_one(tail);
                    tail = dst;
                }
            }
            out_slots[k++] = (int64_t)s.table[pos / bs] * bs + off;
            s.len = pos + 1;
        }
    }
    *num_pairs = np;
    return pkv::ok();
}

pkv_status pkv_seq_len(const pkv_allocator *a, int32_t seq_id, int64_t *len) {
    PKV_CHECK_ARG(a && len, PKV_ERR_INVALID_ARG, "NULL argument");
    Guard g(a->mu);
    PKV_CHECK_ARG(a->live_seq(seq_id), PKV_ERR_OUT_OF_RANGE, "sequence %d is not live", seq_id);
    *len = a->seqs[seq_id].len;
    return pkv::ok();
}

pkv_status pkv_seq_block_table(const pkv_allocator *a, int32_t seq_id, int32_t *out, int32_t capacity,
                               int32_t *n) {
    PKV_CHECK_ARG(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
    Guard g(a->mu);
    PKV_CHECK_ARG(a->live_seq(seq_id), PKV_ERR_OUT_OF_RANGE, "sequence %d is not live", seq_id);
    const auto &t = a->seqs[seq_id].table;
    PKV_CHECK_ARG((int64_t)t.size() <= capacity && (out || t.empty()), PKV_ERR_INVALID_ARG,
                  "capacity %d < %zu blocks", capacity, t.size());
    std::copy(t.begin(), t.end(), out);
    *n = (int32_t)t.size();
    return pkv::ok();
}

pkv_status pkv_seq_fill_tables(const pkv_allocator *a, const int32_t *seq_ids, int32_t n, int32_t *tables,
                               int32_t max_blocks, int32_t *seq_lens) {
    PKV_CHECK_ARG(a && (n == 0 || (seq_ids && tables && seq_lens)) && n >= 0 && max_blocks >= 0,
                  PKV_ERR_INVALID_ARG, "bad argument");
    Guard g(a->mu);
    for (int32_t i = 0; i < n; ++i) {
        PKV_CHECK_ARG(a->live_seq(seq_ids[i]), PKV_ERR_OUT_OF_RANGE, "sequence %d is not live", seq_ids[i]);
        PKV_CHECK_ARG((int64_t)a->seqs[seq_ids[i]].table.size() <= max_blocks, PKV_ERR_SHAPE,
                      "sequence %d holds %zu blocks > max_blocks %d", seq_ids[i],
                      a->seqs[seq_ids[i]].table.size(), max_blocks);
        PKV_CHECK_ARG(a->seqs[seq_ids[i]].len <= INT32_MAX, PKV_ERR_SHAPE, "sequence too long");
    }
    for (int32_t i = 0; i < n; ++i) {
        const auto &s = a->seqs[seq_ids[i]];
        int32_t *row = tables + (int64_t)i * max_blocks;
        std::fill(row, row + max_blocks, -1);
        std::copy(s.table.begin(), s.table.end(), row);
        seq_lens[i] = (int32_t)s.len;
    }
    return pkv::ok();
}

// ---- prefix trie + LRU reclaim ----------------------------------------------

pkv_status pkv_prefix_match(pkv_allocator *a, const int32_t *tokens, int64_t num_tokens, int32_t *out_ids,
                            int32_t capacity, int32_t *num_blocks) {
    PKV_CHECK_ARG(a && num_blocks && num_tokens >= 0 && (tokens || num_tokens == 0) && capacity >= 0 &&
                      (out_ids || capacity == 0),
                  PKV_ERR_INVALID_ARG, "bad argument");
    Guard g(a->mu);
    const int32_t bs = a->block_size;
    int32_t node = 0, n = 0;
    std::vector<int32_t> key(bs);
    for (int64_t j = 0; (j + 1) * bs <= num_tokens && n < capacity; ++j) {
        std::copy(tokens + j * bs, tokens + (j + 1) * bs, key.begin());
        auto it = a->nodes[node].children.find(key);
        if (it == a->nodes[node].children.end()) break;
        node = it->second;
        a->nodes[node].last_used = ++a->clock;
        out_ids[n++] = a->nodes[node].block;
    }
    *num_blocks = n;
    return pkv::ok();
}

pkv_status pkv_seq_create_prefixed(pkv_allocator *a, const int32_t *tokens, int64_t num_tokens, int32_t *seq_id,
                                  int64_t *shared_tokens) {
    PKV_CHECK_ARG(a && seq_id && shared_tokens && num_tokens >= 0 && (tokens || num_tokens == 0),
                  PKV_ERR_INVALID_ARG, "bad argument");
    Guard g(a->mu);
    const int32_t bs = a->block_size;
    int32_t node = 0;
    pkv_allocator::Seq sq;
    std::vector<int32_t> key(bs);
    for (int64_t j = 0; (j + 1) * bs <= num_tokens; ++j) {
        std::copy(tokens + j * bs, tokens + (j + 1) * bs, key.begin());
        auto it = a->nodes[node].children.find(key);
        if (it == a->nodes[node].children.end()) break;
        node = it->second;
        a->nodes[node].last_used = ++a->clock;
        sq.table.push_back(a->nodes[node].block);
    }
    for (int32_t id : sq.table) a->refcount[id] += 1;  // one retain per share
    sq.len = (int64_t)sq.table.size() * bs;
    *shared_tokens = sq.len;
    a->seqs.push_back(std::move(sq));
    *seq_id = (int32_t)a->seqs.size() - 1;
    return pkv::ok();
}

pkv_status pkv_prefix_insert(pkv_allocator *a, const int32_t *tokens, int64_t num_tokens, const int32_t *block_ids,
                             int32_t num_ids) {
    PKV_CHECK_ARG(a && num_tokens >= 0 && num_ids >= 0 && (tokens || num_tokens == 0) && (block_ids || num_ids == 0),
                  PKV_ERR_INVALID_ARG, "bad argument");
    Guard g(a->mu);
    const int32_t bs = a->block_size;
    const int64_t n = std::min<int64_t>(num_ids, num_tokens / bs);
    for (int64_t j = 0; j < n; ++j)
        PKV_CHECK_ARG(a->valid_id(block_ids[j]) && a->refcount[block_ids[j]] > 0, PKV_ERR_DOUBLE_FREE,
                      "block %d is not handed out", block_ids[j]);
    int32_t node = 0;
    for (int64_t j = 0; j < n; ++j) {
        std::vector<int32_t> key(tokens + j * bs, tokens + (j + 1) * bs);
        auto it = a->nodes[node].children.find(key);
        int32_t child;
        if (it == a->nodes[node].children.end()) {
            pkv_allocator::Node nd;
            nd.parent = node;
            nd.key = key;
            nd.block = block_ids[j];
            a->nodes.push_back(std::move(nd));
            child = (int32_t)a->nodes.size() - 1;
            a->nodes[node].children.emplace(std::move(key), child);
            a->refcount[block_ids[j]] += 1;  // the trie's own reference
            a->trie_nodes += 1;
        } else {
            child = it->second;  // first writer wins
        }
        node = child;
        a->nodes[node].last_used = ++a->clock;
    }
    return pkv::ok();
}

pkv_status pkv_prefix_evict(pkv_allocator *a, int32_t max_blocks, int32_t *out_ids, int32_t *num_evicted) {
    PKV_CHECK_ARG(a && num_evicted && max_blocks >= 0 && (out_ids || max_blocks == 0), PKV_ERR_INVALID_ARG,
                  "bad argument");
    Guard g(a->mu);
    int32_t n = 0;
    while (n < max_blocks) {
        // least recently used leaf whose block only the trie still holds (ties: oldest node)
        int32_t best = -1;
        for (int32_t i = 1; i < (int32_t)a->nodes.size(); ++i) {
            const auto &nd = a->nodes[i];
            if (!nd.live || !nd.children.empty() || a->refcount[nd.block] != 1) continue;
            if (best < 0 || nd.last_used < a->nodes[best].last_used) best = i;
        }
        if (best < 0) break;
        auto &nd = a->nodes[best];
        a->nodes[nd.parent].children.erase(nd.key);
        nd.live = false;
        a->trie_nodes -= 1;
        a->release_one(nd.block);
        out_ids[n++] = nd.block;
    }
    *num_evicted = n;
    return pkv::ok();
}

int32_t pkv_prefix_num_nodes(const pkv_allocator *a) {
    if (!a) return -1;
    Guard g(a->mu);
    return a->trie_nodes;
}

pkv_status pkv_check_copy_pairs(const int64_t *p, int32_t num_pairs, int32_t num_blocks) {
    PKV_CHECK_ARG((p || num_pairs == 0) && num_pairs >= 0 && num_blocks > 0, PKV_ERR_INVALID_ARG,
                  "bad argument");
    std::vector<char> is_src(num_blocks, 0), is_dst(num_blocks, 0);
    for (int32_t i = 0; i < num_pairs; ++i) {
        int64_t s = p[2 * i], d = p[2 * i + 1];
        PKV_CHECK_ARG(s >= 0 && s < num_blocks && d >= 0 && d < num_blocks, PKV_ERR_OUT_OF_RANGE,
                      "pair %d (%lld, %lld) outside [0, %d)", i, (long long)s, (long long)d, num_blocks);
        PKV_CHECK_ARG(s != d, PKV_ERR_INVALID_ARG, "pair %d copies block %lld onto itself", i, (long long)s);
        PKV_CHECK_ARG(!is_dst[d], PKV_ERR_INVALID_ARG, "block %lld is a dst twice", (long long)d);
        is_dst[d] = 1;
        is_src[s] = 1;
    }
    for (int32_t i = 0; i < num_pairs; ++i)
        PKV_CHECK_ARG(!is_src[p[2 * i + 1]], PKV_ERR_INVALID_ARG, "block %lld is both a src and a dst",
                      (long long)p[2 * i + 1]);
    return pkv::ok();
}

}  // extern "C"
