// Block pool bookkeeping: free list, refcounts, block tables, fork,
// append with copy-on-write, free.  Host only; device work for appends goes
// through launch_kv_write.
//
// Semantics ("Dendrite" page, section details and its API example; "Trellis"
// page, section "RadixAttention in Trellis"; "SGLang RadixAttention" page,
// reference-counting section):
//   fork      copies the parent's block table and bumps each block's refcount;
//   append    writes into the last block in place when this sequence holds it
//             alone, copies a shared partially-filled last block first
//             (copy-on-write), and takes fresh blocks for the rest;
//   free      drops every refcount by one; blocks at zero return to the pool.
// Allocation order: the free list starts as a Fisher-Yates shuffle of
// [0, NB) driven by splitmix64(alloc_seed) (identity for seed 0): for i from
// NB-1 down to 1, j = next() mod (i+1), swap a[i], a[j].  Allocation takes
// the front, a freed block goes to the front, a freed sequence releases its
// table from the last entry to the first.  Sequence ids: lowest unused id.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/kvp.h"
#include "kvp_internal.h"

struct kvp_pool {
    kvp_pool_desc desc{};
    void *k = nullptr;       // bf16 K/V, or the 4-bit codes of a 4-bit pool
    void *v = nullptr;
    void *k_exp = nullptr;   // 4-bit pool: row exponents
    void *v_exp = nullptr;
    bool kv4 = false;
    std::vector<int32_t> free_;            // back() is the front of the free list
    std::vector<int32_t> ref;
    std::vector<std::vector<int32_t>> tables;
    std::vector<int32_t> lens;
    std::vector<uint8_t> live;
    std::set<int32_t> free_ids;
    int64_t cow_count = 0;
    // scratch reused by appends and exports
    std::vector<int32_t> slots, cow, stage;
};

namespace {

uint64_t splitmix64_next(uint64_t &state) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

bool is_live(const kvp_pool *p, int32_t s) {
    return p && s >= 0 && s < p->desc.max_seqs && p->live[s];
}

int32_t pop_block(kvp_pool *p) {
    int32_t b = p->free_.back();
    p->free_.pop_back();
    p->ref[b] = 1;
    return b;
}

struct Need {
    int cow;
    int64_t fresh;
};

// Blocks an append of ntok tokens to s would take, given refcount drops
// `dec` already implied by earlier appends of the same batch.
Need blocks_needed(const kvp_pool *p, int32_t s, int32_t ntok,
                   const std::unordered_map<int32_t, int32_t> *dec) {
    const int32_t bs = p->desc.block_size;
    const auto &t = p->tables[s];
    const int64_t n = p->lens[s];
    Need need{0, 0};
    if (ntok > 0 && n % bs != 0) {
        int32_t last = t.back();
        int32_t rc = p->ref[last];
        if (dec) {
            auto it = dec->find(last);
            if (it != dec->end()) rc -= it->second;
        }
        need.cow = rc > 1 ? 1 : 0;
    }
    need.fresh = (n + ntok + bs - 1) / bs - (int64_t)t.size();
    return need;
}

// Commits a reserved append: performs the bookkeeping and appends the slot
// ids (block*bs + slot) and any copy-on-write triple to the output vectors.
void commit_append(kvp_pool *p, int32_t s, int32_t ntok, std::vector<int32_t> &slots,
                   std::vector<int32_t> &cow) {
    const int32_t bs = p->desc.block_size;
    auto &t = p->tables[s];
    const int32_t n = p->lens[s];
    const int32_t used = n % bs;
    if (ntok > 0 && used != 0 && p->ref[t.back()] > 1) {
        int32_t old = t.back();
        int32_t nb = pop_block(p);
        p->ref[old] -= 1;
        t.back() = nb;
        cow.push_back(old);
        cow.push_back(nb);
        cow.push_back(used);
        p->cow_count += 1;
    }
    for (int32_t i = 0; i < ntok; ++i) {
        int32_t pos = n + i;
        if (pos % bs == 0) t.push_back(pop_block(p));
        slots.push_back(t[pos / bs] * bs + pos % bs);
    }
    p->lens[s] = n + ntok;
}

int check_append(const kvp_pool *p, int32_t s, int32_t ntok,
                 const std::unordered_map<int32_t, int32_t> *dec, Need *out) {
    if (!is_live(p, s) || ntok < 0) return KVP_ERR_INVALID;
    Need nd = blocks_needed(p, s, ntok, dec);
    if ((int64_t)p->tables[s].size() + nd.fresh > p->desc.max_blocks_per_seq) return KVP_ERR_INVALID;
    if ((int64_t)p->lens[s] + ntok > (int64_t)INT32_MAX / 2) return KVP_ERR_INVALID;
    *out = nd;
    return KVP_OK;
}

// The device write of an append: the copy-on-write triples cow[0..3*ncow)
// and the token scatter to slots[0..ntok).
int issue_write_lists(kvp_pool *p, const int32_t *slots, const int32_t *cow, int32_t ncow, const void *k,
                      const void *v, int32_t ntok, void *stream) {
    if (ntok == 0 && ncow == 0) return KVP_OK;
    if (p->kv4) {
        kvp::Kv4Write w{};
        w.k_codes = p->k;
        w.v_codes = p->v;
        w.k_exp = p->k_exp;
        w.v_exp = p->v_exp;
        w.k = k;
        w.v = v;
        w.L = p->desc.num_layers;
        w.NB = p->desc.num_blocks;
        w.Hkv = p->desc.num_kv_heads;
        w.bs = p->desc.block_size;
        w.d = p->desc.head_dim;
        w.ntok = ntok;
        w.slots = slots;
        w.ncow = ncow;
        w.cow = cow;
        return kvp::launch_kv4_write(w, (cudaStream_t)stream) == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
    }
    kvp::KvWrite w{};
    w.k_pool = p->k;
    w.v_pool = p->v;
    w.k = k;
    w.v = v;
    w.L = p->desc.num_layers;
    w.NB = p->desc.num_blocks;
    w.Hkv = p->desc.num_kv_heads;
    w.bs = p->desc.block_size;
    w.d = p->desc.head_dim;
    w.ntok = ntok;
    w.slots = slots;
    w.ncow = ncow;
    w.cow = cow;
    cudaError_t e = kvp::launch_kv_write(w, (cudaStream_t)stream);
    return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

// The write of the append staged in the pool.
int issue_write(kvp_pool *p, const void *k, const void *v, int32_t ntok, void *stream) {
    return issue_write_lists(p, p->slots.data(), p->cow.data(), (int32_t)(p->cow.size() / 3), k, v, ntok, stream);
}

bool aligned16(const void *ptr) { return ((uintptr_t)ptr & 15) == 0; }


bool desc_valid(const kvp_pool_desc &d) {
    return d.num_layers > 0 && d.num_blocks > 0 && d.block_size > 0 && d.num_kv_heads > 0 && d.head_dim > 0 &&
           d.head_dim % 8 == 0 && d.max_seqs > 0 && d.max_blocks_per_seq > 0 &&
           (int64_t)d.block_size * d.max_blocks_per_seq <= (int64_t)INT32_MAX / 2;
}

kvp_pool *new_pool(const kvp_pool_desc &d) {
    kvp_pool *p = new (std::nothrow) kvp_pool();
    if (!p) return nullptr;
    p->desc = d;
    std::vector<int32_t> a(d.num_blocks);
    for (int32_t i = 0; i < d.num_blocks; ++i) a[i] = i;
    if (d.alloc_seed != 0) {
        uint64_t st = d.alloc_seed;
        for (int64_t i = d.num_blocks - 1; i >= 1; --i) {
            uint64_t j = splitmix64_next(st) % (uint64_t)(i + 1);
            std::swap(a[i], a[j]);
        }
    }
    p->free_.assign(a.rbegin(), a.rend());
    p->ref.assign(d.num_blocks, 0);
    p->tables.resize(d.max_seqs);
    p->lens.assign(d.max_seqs, 0);
    p->live.assign(d.max_seqs, 0);
    for (int32_t i = 0; i < d.max_seqs; ++i) p->free_ids.insert(i);
    return p;
}

}  // namespace

extern "C" {

int kv_pool_create(const kvp_pool_desc *desc, void *k_storage, void *v_storage, kvp_pool **out) {
    if (!desc || !out || !desc_valid(*desc)) return KVP_ERR_INVALID;
    if ((k_storage == nullptr) != (v_storage == nullptr)) return KVP_ERR_INVALID;
    if (k_storage && (!aligned16(k_storage) || !aligned16(v_storage))) return KVP_ERR_INVALID;
    kvp_pool *p = new_pool(*desc);
    if (!p) return KVP_ERR_OOM;
    p->k = k_storage;
    p->v = v_storage;
    *out = p;
    return KVP_OK;
}

int kv_pool_create_kv4(const kvp_pool_desc *desc, void *k_codes, void *k_exps, void *v_codes, void *v_exps,
                       kvp_pool **out) {
    if (!desc || !out || !desc_valid(*desc)) return KVP_ERR_INVALID;
    const kvp_pool_desc &d = *desc;
    // 16-byte code rows (d/2 bytes) and whole 16-byte groups of exponents per block
    if ((d.head_dim != 64 && d.head_dim != 128) || d.block_size % 16 != 0) return KVP_ERR_INVALID;
    if (!k_codes || !k_exps || !v_codes || !v_exps) return KVP_ERR_INVALID;
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_exps) || !aligned16(v_exps))
        return KVP_ERR_INVALID;
    kvp_pool *p = new_pool(d);
    if (!p) return KVP_ERR_OOM;
    p->k = k_codes;
    p->v = v_codes;
    p->k_exp = k_exps;
    p->v_exp = v_exps;
    p->kv4 = true;
    *out = p;
    return KVP_OK;
}

int kv_pool_destroy(kvp_pool *pool) {
    if (!pool) return KVP_ERR_INVALID;
    delete pool;
    return KVP_OK;
}

int seq_alloc(kvp_pool *p, int32_t *seq_out) {
    if (!p || !seq_out) return KVP_ERR_INVALID;
    if (p->free_ids.empty()) return KVP_ERR_OOM;
    int32_t s = *p->free_ids.begin();
    p->free_ids.erase(p->free_ids.begin());
    p->live[s] = 1;
    p->tables[s].clear();
    p->lens[s] = 0;
    *seq_out = s;
    return KVP_OK;
}

int seq_fork(kvp_pool *p, int32_t parent, int32_t *child_out) {
    if (!p || !child_out || !is_live(p, parent)) return KVP_ERR_INVALID;
    if (p->free_ids.empty()) return KVP_ERR_OOM;
    int32_t s = *p->free_ids.begin();
    p->free_ids.erase(p->free_ids.begin());
    p->live[s] = 1;
    p->tables[s] = p->tables[parent];
    p->lens[s] = p->lens[parent];
    for (int32_t b : p->tables[s]) p->ref[b] += 1;
    *child_out = s;
    return KVP_OK;
}

int seq_accept_draft(kvp_pool *p, int32_t seq, int32_t ctx_len, const int32_t *parent, int32_t n_draft,
                     int32_t accepted, int32_t *path_out, int32_t *n_path_out, void *stream) {
    if (!is_live(p, seq) || ctx_len < 0 || n_draft < 0 || n_draft > kvp::kMaxDraft) return KVP_ERR_INVALID;
    if ((int64_t)ctx_len + n_draft != p->lens[seq] || accepted < -1 || accepted >= n_draft) return KVP_ERR_INVALID;
    if (n_draft > 0 && !parent) return KVP_ERR_INVALID;
    for (int32_t i = 0; i < n_draft; ++i)
        if (parent[i] < -1 || parent[i] >= i) return KVP_ERR_INVALID;
    // the accepted path, root first
    int32_t path[kvp::kMaxDraft];
    int32_t np = 0;
    for (int32_t j = accepted; j >= 0; j = parent[j]) path[np++] = j;
    std::reverse(path, path + np);
    const int32_t bs = p->desc.block_size;
    auto &t = p->tables[seq];
    // blocks that receive a moved token and are shared: copied first
    std::vector<int32_t> shared;
    for (int32_t i = 0; i < np; ++i) {
        if (path[i] == i) continue;
        const int32_t j = (ctx_len + i) / bs;
        if (p->ref[t[j]] > 1 && (shared.empty() || shared.back() != j)) shared.push_back(j);
    }
    if ((int64_t)shared.size() > (int64_t)p->free_.size()) return KVP_ERR_OOM;
    p->cow.clear();
    for (int32_t j : shared) {
        const int32_t old = t[j], fresh = pop_block(p);
        p->ref[old] -= 1;
        t[j] = fresh;
        p->cow_count += 1;
        p->cow.push_back(old);
        p->cow.push_back(fresh);
    }
    p->slots.clear();   // source slots
    p->stage.clear();   // destination slots
    for (int32_t i = 0; i < np; ++i) {
        if (path[i] == i) continue;
        const int32_t sp = ctx_len + path[i], dp = ctx_len + i;
        p->slots.push_back(t[sp / bs] * bs + sp % bs);
        p->stage.push_back(t[dp / bs] * bs + dp % bs);
    }
    int rc = KVP_OK;
    if (p->k && p->kv4 && (!p->cow.empty() || !p->slots.empty())) {
        kvp::Kv4Move m{};
        m.k_codes = p->k;
        m.v_codes = p->v;
        m.k_exp = p->k_exp;
        m.v_exp = p->v_exp;
        m.L = p->desc.num_layers;
        m.NB = p->desc.num_blocks;
        m.Hkv = p->desc.num_kv_heads;
        m.bs = bs;
        m.d = p->desc.head_dim;
        m.ncow = (int32_t)shared.size();
        m.cow = p->cow.data();
        m.nmove = (int32_t)p->slots.size();
        m.src = p->slots.data();
        m.dst = p->stage.data();
        if (kvp::launch_kv4_move(m, (cudaStream_t)stream) != cudaSuccess) rc = KVP_ERR_CUDA;
    } else if (p->k && (!p->cow.empty() || !p->slots.empty())) {
        kvp::KvMove m{};
        m.k_pool = p->k;
        m.v_pool = p->v;
        m.L = p->desc.num_layers;
        m.NB = p->desc.num_blocks;
        m.Hkv = p->desc.num_kv_heads;
        m.bs = bs;
        m.d = p->desc.head_dim;
        m.ncow = (int32_t)shared.size();
        m.cow = p->cow.data();
        m.nmove = (int32_t)p->slots.size();
        m.src = p->slots.data();
        m.dst = p->stage.data();
        if (kvp::launch_kv_move(m, (cudaStream_t)stream) != cudaSuccess) rc = KVP_ERR_CUDA;
    }
    // release the blocks past the new end, last first
    const int32_t new_len = ctx_len + np;
    const size_t keep = (size_t)((new_len + bs - 1) / bs);
    for (size_t j = t.size(); j-- > keep;)
        if (--p->ref[t[j]] == 0) p->free_.push_back(t[j]);
    t.resize(keep);
    p->lens[seq] = new_len;
    if (path_out) std::copy(path, path + np, path_out);
    if (n_path_out) *n_path_out = np;
    return rc;
}

int seq_alloc_prefix(kvp_pool *p, const int32_t *blocks, int32_t n_blocks, int32_t *seq_out) {
    if (!p || !seq_out || n_blocks < 0 || (n_blocks > 0 && !blocks)) return KVP_ERR_INVALID;
    if (n_blocks > p->desc.max_blocks_per_seq) return KVP_ERR_INVALID;
    for (int32_t i = 0; i < n_blocks; ++i)
        if (blocks[i] < 0 || blocks[i] >= p->desc.num_blocks || p->ref[blocks[i]] <= 0) return KVP_ERR_INVALID;
    if (p->free_ids.empty()) return KVP_ERR_OOM;
    int32_t s = *p->free_ids.begin();
    p->free_ids.erase(p->free_ids.begin());
    p->live[s] = 1;
    p->tables[s].assign(blocks, blocks + n_blocks);
    p->lens[s] = n_blocks * p->desc.block_size;
    for (int32_t i = 0; i < n_blocks; ++i) p->ref[blocks[i]] += 1;
    *seq_out = s;
    return KVP_OK;
}

int seq_free(kvp_pool *p, int32_t seq) {
    if (!is_live(p, seq)) return KVP_ERR_INVALID;
    auto &t = p->tables[seq];
    for (auto it = t.rbegin(); it != t.rend(); ++it) {
        if (--p->ref[*it] == 0) p->free_.push_back(*it);
    }
    t.clear();
    t.shrink_to_fit();
    p->lens[seq] = 0;
    p->live[seq] = 0;
    p->free_ids.insert(seq);
    return KVP_OK;
}

int seq_reserve(kvp_pool *p, int32_t seq, int32_t ntok, int32_t *slots_out, int32_t *cow_out) {
    if (!p) return KVP_ERR_INVALID;
    Need nd{};
    int rc = check_append(p, seq, ntok, nullptr, &nd);
    if (rc) return rc;
    if (nd.cow + nd.fresh > (int64_t)p->free_.size()) return KVP_ERR_OOM;
    p->slots.clear();
    p->cow.clear();
    commit_append(p, seq, ntok, p->slots, p->cow);
    if (slots_out) std::memcpy(slots_out, p->slots.data(), sizeof(int32_t) * (size_t)ntok);
    if (cow_out) {
        if (p->cow.empty()) {
            cow_out[0] = -1; cow_out[1] = -1; cow_out[2] = 0;
        } else {
            std::memcpy(cow_out, p->cow.data(), sizeof(int32_t) * 3);
        }
    }
    return KVP_OK;
}

int seq_append(kvp_pool *p, int32_t seq, const void *k, const void *v, int32_t ntok, void *stream) {
    if (!p) return KVP_ERR_INVALID;
    if (!p->k) return KVP_ERR_STATE;
    if (ntok > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return KVP_ERR_INVALID;
    Need nd{};
    int rc = check_append(p, seq, ntok, nullptr, &nd);
    if (rc) return rc;
    if (nd.cow + nd.fresh > (int64_t)p->free_.size()) return KVP_ERR_OOM;
    p->slots.clear();
    p->cow.clear();
    commit_append(p, seq, ntok, p->slots, p->cow);
    return issue_write(p, k, v, ntok, stream);
}

int seq_append_batch(kvp_pool *p, int32_t nseq, const int32_t *seqs, const int32_t *ntoks,
                     const void *k, const void *v, void *stream) {
    int32_t total = 0;
    int rc = kvp::append_batch_commit(p, nseq, seqs, ntoks, k, v, &total);
    if (rc) return rc;
    return issue_write(p, k, v, total, stream);
}

int seq_block_table(const kvp_pool *p, int32_t seq, int32_t *host_out, int32_t cap,
                    int32_t *nblocks_out) {
    if (!is_live(p, seq)) return KVP_ERR_INVALID;
    const auto &t = p->tables[seq];
    if (host_out && cap < (int32_t)t.size()) return KVP_ERR_INVALID;
    if (host_out && !t.empty()) std::memcpy(host_out, t.data(), sizeof(int32_t) * t.size());
    if (nblocks_out) *nblocks_out = (int32_t)t.size();
    return KVP_OK;
}

int seq_len(const kvp_pool *p, int32_t seq, int32_t *len_out) {
    if (!is_live(p, seq) || !len_out) return KVP_ERR_INVALID;
    *len_out = p->lens[seq];
    return KVP_OK;
}

int block_refcount(const kvp_pool *p, int32_t block, int32_t *rc_out) {
    if (!p || !rc_out || block < 0 || block >= p->desc.num_blocks) return KVP_ERR_INVALID;
    *rc_out = p->ref[block];
    return KVP_OK;
}

int kvp_free_block_count(const kvp_pool *p, int32_t *n_out) {
    if (!p || !n_out) return KVP_ERR_INVALID;
    *n_out = (int32_t)p->free_.size();
    return KVP_OK;
}

int kvp_cow_count(const kvp_pool *p, int64_t *n_out) {
    if (!p || !n_out) return KVP_ERR_INVALID;
    *n_out = p->cow_count;
    return KVP_OK;
}

int kvp_gather_tables(const kvp_pool *p, const int32_t *seqs, int32_t n, int32_t width,
                      int32_t *h_tables, int32_t *h_lens) {
    if (!p || n < 0 || width < 0 || (n > 0 && !seqs)) return KVP_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) {
        if (!is_live(p, seqs[i])) return KVP_ERR_INVALID;
        if (h_tables && (int32_t)p->tables[seqs[i]].size() > width) return KVP_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        const auto &t = p->tables[seqs[i]];
        if (h_tables) {
            int32_t *row = h_tables + (size_t)i * width;
            std::fill(row, row + width, -1);
            if (!t.empty()) std::memcpy(row, t.data(), sizeof(int32_t) * t.size());
        }
        if (h_lens) h_lens[i] = p->lens[seqs[i]];
    }
    return KVP_OK;
}

int kvp_export_tables(kvp_pool *p, const int32_t *seqs, int32_t n, int32_t width,
                      int32_t *d_tables, int32_t *d_lens, void *stream) {
    if (!p || n < 0 || width < 0) return KVP_ERR_INVALID;
    p->stage.assign((size_t)n * width + n, -1);
    int rc = kvp_gather_tables(p, seqs, n, width, p->stage.data(), p->stage.data() + (size_t)n * width);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (d_tables && n * width > 0 &&
        cudaMemcpyAsync(d_tables, p->stage.data(), sizeof(int32_t) * (size_t)n * width,
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    if (d_lens && n > 0 &&
        cudaMemcpyAsync(d_lens, p->stage.data() + (size_t)n * width, sizeof(int32_t) * (size_t)n,
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    // pageable source: the copy is staged before return, so `stage` may be reused
    return KVP_OK;
}

const char *kvp_strerror(int code) {
    switch (code) {
        case KVP_OK: return "ok";
        case KVP_ERR_INVALID: return "invalid argument";
        case KVP_ERR_OOM: return "out of blocks or sequence slots";
        case KVP_ERR_STATE: return "operation not possible in this state";
        case KVP_ERR_CUDA: return "CUDA runtime error";
        case KVP_ERR_DEVICE: return "device-side check failed";
        case KVP_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown error";
    }
}

}  // extern "C"

namespace kvp {

int32_t pool_block_size(const kvp_pool *p) { return p->desc.block_size; }
int32_t pool_num_blocks(const kvp_pool *p) { return p->desc.num_blocks; }
int32_t pool_free_count(const kvp_pool *p) { return (int32_t)p->free_.size(); }
bool pool_block_in_use(const kvp_pool *p, int32_t b) {
    return b >= 0 && b < p->desc.num_blocks && p->ref[b] > 0;
}
void pool_hold_block(kvp_pool *p, int32_t b) { p->ref[b] += 1; }
bool pool_drop_block(kvp_pool *p, int32_t b) {
    if (--p->ref[b] != 0) return false;
    p->free_.push_back(b);   // the front of the free list
    return true;
}

int append_batch_check(kvp_pool *p, int32_t nseq, const int32_t *seqs, const int32_t *ntoks,
                       int64_t *total_out) {
    if (total_out) *total_out = 0;
    if (!p || nseq < 0 || (nseq > 0 && (!seqs || !ntoks))) return KVP_ERR_INVALID;
    if (!p->k) return KVP_ERR_STATE;
    std::unordered_map<int32_t, int32_t> dec;
    std::set<int32_t> seen;
    int64_t need = 0, total = 0;
    for (int32_t i = 0; i < nseq; ++i) {
        if (!seen.insert(seqs[i]).second) return KVP_ERR_INVALID;
        Need nd{};
        int rc = check_append(p, seqs[i], ntoks[i], &dec, &nd);
        if (rc) return rc;
        if (nd.cow) dec[p->tables[seqs[i]].back()] += 1;
        need += nd.cow + nd.fresh;
        total += ntoks[i];
    }
    if (total > INT32_MAX / 2) return KVP_ERR_INVALID;
    if (total_out) *total_out = total;
    if (need > (int64_t)p->free_.size()) return KVP_ERR_OOM;
    return KVP_OK;
}

int append_batch_commit(kvp_pool *p, int32_t nseq, const int32_t *seqs, const int32_t *ntoks, const void *k,
                        const void *v, int32_t *total_out) {
    int64_t total = 0;
    int rc = append_batch_check(p, nseq, seqs, ntoks, &total);
    if (rc != KVP_OK && rc != KVP_ERR_OOM) return rc;
    if (total > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return KVP_ERR_INVALID;
    if (rc) return rc;
    p->slots.clear();
    p->cow.clear();
    for (int32_t i = 0; i < nseq; ++i) commit_append(p, seqs[i], ntoks[i], p->slots, p->cow);
    *total_out = (int32_t)total;
    return KVP_OK;
}

int append_batch_commit_lists(kvp_pool *p, int32_t nseq, const int32_t *seqs, const int32_t *ntoks,
                              std::vector<int32_t> &slots, std::vector<int32_t> &cow, int32_t *total_out) {
    int64_t total = 0;
    int rc = append_batch_check(p, nseq, seqs, ntoks, &total);
    if (rc) return rc;
    slots.clear();
    cow.clear();
    for (int32_t i = 0; i < nseq; ++i) commit_append(p, seqs[i], ntoks[i], slots, cow);
    *total_out = (int32_t)total;
    return KVP_OK;
}

int append_issue_lists(kvp_pool *p, const std::vector<int32_t> &slots, const std::vector<int32_t> &cow,
                       const void *k, const void *v, void *stream) {
    return issue_write_lists(p, slots.data(), cow.data(), (int32_t)(cow.size() / 3), k, v, (int32_t)slots.size(),
                             stream);
}

PoolView pool_view(const kvp_pool *p) {
    const kvp_pool_desc &d = p->desc;
    return PoolView{d.num_layers, d.num_blocks, d.block_size, d.num_kv_heads, d.head_dim,
                    p->k, p->v, p->k_exp, p->v_exp, p->kv4};
}

int pool_tables(const kvp_pool *p, const int32_t *seqs, int32_t n, int32_t *width, int32_t **tables,
                int32_t **lens) {
    if (!p || n <= 0 || !seqs) return KVP_ERR_INVALID;
    int32_t w = 1;
    for (int32_t i = 0; i < n; ++i) {
        if (!is_live(p, seqs[i])) return KVP_ERR_INVALID;
        w = std::max(w, (int32_t)p->tables[seqs[i]].size());
    }
    // the pool's scratch: valid until the next call on this pool
    auto &st = const_cast<kvp_pool *>(p)->stage;
    st.assign((size_t)n * w + n, -1);
    int rc = kvp_gather_tables(p, seqs, n, w, st.data(), st.data() + (size_t)n * w);
    if (rc) return rc;
    *width = w;
    *tables = st.data();
    *lens = st.data() + (size_t)n * w;
    return KVP_OK;
}

}  // namespace kvp
