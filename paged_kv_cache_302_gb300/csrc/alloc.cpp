// alloc.cpp -- host block allocator behind pa_alloc_* (pa.h).
//
// PagedAttention explainer (0h-n0.github.io, arXiv 2309.06180):
//  * 技術的詳細 / PagedAttentionアルゴリズム: a sequence of T tokens occupies
//    ceil(T/B) blocks placed anywhere; a per-sequence table maps logical to
//    physical blocks.
//  * Copy-on-Write KVキャッシュ共有: shared blocks carry a reference count; a
//    write into a block whose count is above one copies the block first.
//  * 実装のポイント: one slab managed by the library's own allocator; blocks are
//    taken on demand and returned when a request ends.
// The free list is a LIFO stack; every call validates first and then applies,
// so a failing call leaves the state unchanged.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pa_internal.h"

namespace pa {

struct Seq {
    std::vector<int32_t> blocks;
    int64_t ntok = 0;
};

struct Allocator {
    int NB = 0, B = 0;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> ref;
    std::unordered_map<int, Seq> seqs;
};

static Allocator* as_alloc(void* h) { return static_cast<Allocator*>(h); }

// Blocks a single-sequence append of n tokens takes from the free list, given
// the current reference count `last_ref` of its last block.
static int64_t blocks_needed(const Allocator& A, const Seq& s, int64_t n, int last_ref) {
    if (n <= 0) return 0;
    int64_t need = 0;
    if (s.ntok % A.B != 0 && last_ref > 1) need += 1;  // copy-on-write of the shared partial block
    const int64_t have = (s.ntok + A.B - 1) / A.B;
    const int64_t want = (s.ntok + n + A.B - 1) / A.B;
    return need + (want - have);
}

// Applies an append whose block demand has been checked.  Every table entry
// the append sets (a new block, or the copy that replaces a shared one) is
// recorded in `upd` as (row, logical block, physical block) when upd != NULL.
static void apply_append(Allocator& A, Seq& s, int64_t n, int64_t* slots, std::vector<int64_t>& cow,
                         std::vector<int32_t>* upd = nullptr, int row = 0) {
    for (int64_t i = 0; i < n; ++i) {
        const int64_t pos = s.ntok;
        const int64_t off = pos % A.B;
        if (off == 0) {
            const int32_t b = A.free_stack.back();
            A.free_stack.pop_back();
            A.ref[b] = 1;
            s.blocks.push_back(b);
            if (upd) upd->insert(upd->end(), {row, (int32_t)(pos / A.B), b});
        } else if (A.ref[s.blocks.back()] > 1) {
            const int32_t old = s.blocks.back();
            const int32_t b = A.free_stack.back();
            A.free_stack.pop_back();
            A.ref[b] = 1;
            A.ref[old] -= 1;
            s.blocks.back() = b;
            cow.push_back(old);
            cow.push_back(b);
            if (upd) upd->insert(upd->end(), {row, (int32_t)(pos / A.B), b});
        }
        slots[i] = (int64_t)s.blocks[pos / A.B] * A.B + off;
        s.ntok = pos + 1;
    }
}

}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_alloc_create(int NB, int B, const int32_t* initial_free_order, void** out) {
    if (!out) return fail(PA_ERR_INVALID, "out is null");
    *out = nullptr;
    if (NB <= 0 || B <= 0) return fail(PA_ERR_INVALID, "NB and B must be positive");
    Allocator* A = new (std::nothrow) Allocator;
    if (!A) return fail(PA_ERR_OOM, "host allocation failed");
    A->NB = NB;
    A->B = B;
    A->ref.assign(NB, 0);
    A->free_stack.resize(NB);
    if (initial_free_order) {
        std::vector<char> seen(NB, 0);
        for (int i = 0; i < NB; ++i) {
            const int32_t b = initial_free_order[i];
            if (b < 0 || b >= NB || seen[b]) {
                delete A;
                return fail(PA_ERR_INVALID, "initial_free_order must be a permutation of 0..NB-1");
            }
            seen[b] = 1;
            A->free_stack[NB - 1 - i] = b;
        }
    } else {
        for (int i = 0; i < NB; ++i) A->free_stack[NB - 1 - i] = i;
    }
    *out = A;
    return PA_OK;
}

void pa_alloc_destroy(void* alloc) { delete as_alloc(alloc); }

pa_status pa_alloc_add_seq(void* alloc, int seq_id) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    if (seq_id < 0) return fail(PA_ERR_INVALID, "seq_id must be >= 0");
    if (A->seqs.count(seq_id)) return fail(PA_ERR_INVALID, "sequence %d exists", seq_id);
    A->seqs.emplace(seq_id, Seq());
    return PA_OK;
}

pa_status pa_alloc_append_slots(void* alloc, int seq_id, int n, int64_t* slots_out, int64_t* cow_pairs_out,
                                int cow_cap, int* n_cow) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    auto it = A->seqs.find(seq_id);
    if (it == A->seqs.end()) return fail(PA_ERR_INVALID, "unknown sequence %d", seq_id);
    if (n < 0) return fail(PA_ERR_INVALID, "negative token count");
    if (n > 0 && !slots_out) return fail(PA_ERR_INVALID, "slots_out is null");
    Seq& s = it->second;
    const int last_ref = s.blocks.empty() ? 0 : A->ref[s.blocks.back()];
    const int64_t need = blocks_needed(*A, s, n, last_ref);
    const bool will_copy = n > 0 && s.ntok % A->B != 0 && last_ref > 1;
    if (will_copy && (cow_cap < 1 || !cow_pairs_out)) return fail(PA_ERR_INVALID, "cow_pairs_out too small");
    if (need > (int64_t)A->free_stack.size())
        return fail(PA_ERR_OOM, "need %lld blocks, %zu free", (long long)need, A->free_stack.size());
    std::vector<int64_t> cow;
    apply_append(*A, s, n, slots_out, cow);
    for (size_t i = 0; i < cow.size(); ++i) cow_pairs_out[i] = cow[i];
    if (n_cow) *n_cow = (int)(cow.size() / 2);
    return PA_OK;
}

pa_status pa_alloc_append_batch(void* alloc, int n_seqs, const int32_t* seq_ids, const int32_t* n_tokens,
                                int64_t* slots_out, int64_t* cow_pairs_out, int cow_cap, int* n_cow,
                                int32_t* table_updates_out, int upd_cap, int* n_upd) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    if (n_seqs < 0) return fail(PA_ERR_INVALID, "negative n_seqs");
    if (n_seqs > 0 && (!seq_ids || !n_tokens)) return fail(PA_ERR_INVALID, "null argument");
    // validate and count demand, following the reference counts the earlier
    // sequences of the batch change
    std::unordered_set<int> seen;
    std::unordered_map<int32_t, int> ref_delta;
    int64_t need = 0, total_tok = 0, copies = 0;
    std::vector<Seq*> seqs(n_seqs);
    for (int i = 0; i < n_seqs; ++i) {
        auto it = A->seqs.find(seq_ids[i]);
        if (it == A->seqs.end()) return fail(PA_ERR_INVALID, "unknown sequence %d", seq_ids[i]);
        if (!seen.insert(seq_ids[i]).second) return fail(PA_ERR_INVALID, "sequence %d repeated", seq_ids[i]);
        if (n_tokens[i] < 0) return fail(PA_ERR_INVALID, "negative token count");
        Seq& s = it->second;
        seqs[i] = &s;
        int last_ref = 0;
        if (!s.blocks.empty()) last_ref = A->ref[s.blocks.back()] + ref_delta[s.blocks.back()];
        need += blocks_needed(*A, s, n_tokens[i], last_ref);
        if (n_tokens[i] > 0 && s.ntok % A->B != 0 && last_ref > 1) {
            ref_delta[s.blocks.back()] -= 1;
            copies += 1;
        }
        total_tok += n_tokens[i];
    }
    if (total_tok > 0 && !slots_out) return fail(PA_ERR_INVALID, "slots_out is null");
    if (copies > 0 && (cow_cap < copies || !cow_pairs_out)) return fail(PA_ERR_INVALID, "cow_pairs_out too small");
    if (need > (int64_t)A->free_stack.size())
        return fail(PA_ERR_OOM, "need %lld blocks, %zu free", (long long)need, A->free_stack.size());
    // every table entry set by the batch is a block taken from the free list
    if (table_updates_out && need > upd_cap)
        return fail(PA_ERR_INVALID, "table_updates_out holds %d entries, the batch sets %lld", upd_cap,
                    (long long)need);
    std::vector<int64_t> cow;
    std::vector<int32_t> upd;
    int64_t off = 0;
    for (int i = 0; i < n_seqs; ++i) {
        apply_append(*A, *seqs[i], n_tokens[i], slots_out + off, cow, table_updates_out ? &upd : nullptr, i);
        off += n_tokens[i];
    }
    for (size_t i = 0; i < cow.size(); ++i) cow_pairs_out[i] = cow[i];
    if (n_cow) *n_cow = (int)(cow.size() / 2);
    if (table_updates_out && !upd.empty()) std::memcpy(table_updates_out, upd.data(), upd.size() * sizeof(int32_t));
    if (n_upd) *n_upd = (int)(upd.size() / 3);
    return PA_OK;
}

pa_status pa_alloc_fork(void* alloc, int parent, int child) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    auto it = A->seqs.find(parent);
    if (it == A->seqs.end()) return fail(PA_ERR_INVALID, "unknown sequence %d", parent);
    if (child < 0 || A->seqs.count(child)) return fail(PA_ERR_INVALID, "child %d exists or is negative", child);
    Seq c = it->second;
    for (int32_t b : c.blocks) A->ref[b] += 1;
    A->seqs.emplace(child, std::move(c));
    return PA_OK;
}

pa_status pa_alloc_free_seq(void* alloc, int seq_id) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    auto it = A->seqs.find(seq_id);
    if (it == A->seqs.end()) return fail(PA_ERR_INVALID, "unknown sequence %d", seq_id);
    for (int32_t b : it->second.blocks)
        if (A->ref[b] <= 0) return fail(PA_ERR_STATE, "block %d has no reference", b);
    for (int32_t b : it->second.blocks) {
        if (--A->ref[b] == 0) A->free_stack.push_back(b);
    }
    A->seqs.erase(it);
    return PA_OK;
}

pa_status pa_alloc_block_table(void* alloc, int seq_id, int32_t* out, int cap, int* n) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    auto it = A->seqs.find(seq_id);
    if (it == A->seqs.end()) return fail(PA_ERR_INVALID, "unknown sequence %d", seq_id);
    const auto& bl = it->second.blocks;
    if (n) *n = (int)bl.size();
    if ((int)bl.size() > cap || (!out && !bl.empty())) return fail(PA_ERR_INVALID, "capacity %d < %zu", cap, bl.size());
    if (!bl.empty()) std::memcpy(out, bl.data(), bl.size() * sizeof(int32_t));
    return PA_OK;
}

pa_status pa_alloc_block_tables(void* alloc, int n_seqs, const int32_t* seq_ids, int32_t* out, int MB,
                                int32_t* ctx_out) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    if (n_seqs < 0 || MB <= 0) return fail(PA_ERR_INVALID, "bad sizes");
    if (n_seqs > 0 && (!seq_ids || !out)) return fail(PA_ERR_INVALID, "null argument");
    for (int i = 0; i < n_seqs; ++i) {
        auto it = A->seqs.find(seq_ids[i]);
        if (it == A->seqs.end()) return fail(PA_ERR_INVALID, "unknown sequence %d", seq_ids[i]);
        if ((int64_t)it->second.blocks.size() > MB)
            return fail(PA_ERR_INVALID, "sequence %d has %zu blocks > MB %d", seq_ids[i], it->second.blocks.size(), MB);
    }
    for (int i = 0; i < n_seqs; ++i) {
        const Seq& s = A->seqs.find(seq_ids[i])->second;
        int32_t* row = out + (size_t)i * MB;
        std::copy(s.blocks.begin(), s.blocks.end(), row);
        std::fill(row + s.blocks.size(), row + MB, -1);
        if (ctx_out) ctx_out[i] = (int32_t)s.ntok;
    }
    return PA_OK;
}

pa_status pa_alloc_seq_len(void* alloc, int seq_id, int64_t* out) {
    Allocator* A = as_alloc(alloc);
    if (!A || !out) return fail(PA_ERR_INVALID, "null argument");
    auto it = A->seqs.find(seq_id);
    if (it == A->seqs.end()) return fail(PA_ERR_INVALID, "unknown sequence %d", seq_id);
    *out = it->second.ntok;
    return PA_OK;
}

pa_status pa_alloc_refcount(void* alloc, int block, int* out) {
    Allocator* A = as_alloc(alloc);
    if (!A || !out) return fail(PA_ERR_INVALID, "null argument");
    if (block < 0 || block >= A->NB) return fail(PA_ERR_INVALID, "block %d out of range", block);
    *out = A->ref[block];
    return PA_OK;
}

int pa_alloc_num_free(void* alloc) {
    Allocator* A = as_alloc(alloc);
    return A ? (int)A->free_stack.size() : -1;
}

pa_status pa_alloc_free_list(void* alloc, int32_t* out, int cap, int* n) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    const int sz = (int)A->free_stack.size();
    if (n) *n = sz;
    if (sz > cap || (!out && sz)) return fail(PA_ERR_INVALID, "capacity %d < %d", cap, sz);
    for (int i = 0; i < sz; ++i) out[i] = A->free_stack[sz - 1 - i];
    return PA_OK;
}

// ----------------------------------------------------------------------------- state export / import

static constexpr int64_t kStateMagic = 0x3141415043;  // tags the flat state layout below

pa_status pa_alloc_export(void* alloc, int64_t* out, size_t cap, size_t* n) {
    Allocator* A = as_alloc(alloc);
    if (!A) return fail(PA_ERR_INVALID, "null allocator");
    std::vector<int> ids;
    ids.reserve(A->seqs.size());
    size_t need = 5 + A->free_stack.size() + (size_t)A->NB;
    for (const auto& kv : A->seqs) {
        ids.push_back(kv.first);
        need += 3 + kv.second.blocks.size();
    }
    if (n) *n = need;
    if (!out) return PA_OK;
    if (cap < need) return fail(PA_ERR_INVALID, "capacity %zu < %zu words", cap, need);
    std::sort(ids.begin(), ids.end());
    size_t w = 0;
    out[w++] = kStateMagic;
    out[w++] = A->NB;
    out[w++] = A->B;
    out[w++] = (int64_t)A->free_stack.size();
    out[w++] = (int64_t)ids.size();
    for (int32_t b : A->free_stack) out[w++] = b;  // bottom of the stack first
    for (int32_t r : A->ref) out[w++] = r;
    for (int id : ids) {
        const Seq& q = A->seqs.at(id);
        out[w++] = id;
        out[w++] = q.ntok;
        out[w++] = (int64_t)q.blocks.size();
        for (int32_t b : q.blocks) out[w++] = b;
    }
    return PA_OK;
}

pa_status pa_alloc_import(const int64_t* in, size_t n, void** out) {
    if (!in || !out) return fail(PA_ERR_INVALID, "null argument");
    *out = nullptr;
    if (n < 5 || in[0] != kStateMagic) return fail(PA_ERR_INVALID, "not an allocator state");
    const int64_t NB = in[1], B = in[2], nfree = in[3], nseq = in[4];
    if (NB <= 0 || NB > INT32_MAX || B <= 0 || B > INT32_MAX || nfree < 0 || nfree > NB || nseq < 0)
        return fail(PA_ERR_INVALID, "bad header");
    size_t r = 5;
    if ((size_t)(n - r) < (size_t)nfree + (size_t)NB) return fail(PA_ERR_INVALID, "truncated state");
    Allocator* A = new (std::nothrow) Allocator;
    if (!A) return fail(PA_ERR_OOM, "allocator handle");
    A->NB = (int)NB;
    A->B = (int)B;
    A->free_stack.assign(in + r, in + r + nfree);
    r += nfree;
    A->ref.assign(in + r, in + r + NB);
    r += NB;
    // every block is either free (once, count 0) or counted exactly as often as the tables name it
    std::vector<int64_t> seen(NB, 0);
    auto bad = [&](const char* why) {
        delete A;
        return fail(PA_ERR_INVALID, "inconsistent allocator state: %s", why);
    };
    for (int32_t b : A->free_stack) {
        if (b < 0 || b >= NB || A->ref[b] != 0 || seen[b]) return bad("free list");
        seen[b] = -1;
    }
    for (int64_t i = 0; i < nseq; ++i) {
        if (n - r < 3) return bad("truncated sequence");
        const int64_t id = in[r], ntok = in[r + 1], nb = in[r + 2];
        r += 3;
        if (id < 0 || id > INT32_MAX || ntok < 0 || nb != (ntok + B - 1) / B || (size_t)nb > n - r)
            return bad("sequence header");
        Seq q;
        q.ntok = ntok;
        for (int64_t j = 0; j < nb; ++j) {
            const int64_t b = in[r + j];
            if (b < 0 || b >= NB || seen[b] < 0) return bad("table entry");
            ++seen[b];
            q.blocks.push_back((int32_t)b);
        }
        r += nb;
        if (!A->seqs.emplace((int)id, std::move(q)).second) return bad("duplicate sequence");
    }
    if (r != n) return bad("trailing words");
    for (int64_t b = 0; b < NB; ++b) {
        if (seen[b] == 0) return bad("a block neither free nor in a table");
        if (seen[b] > 0 && seen[b] != A->ref[b]) return bad("reference count");
    }
    *out = A;
    return PA_OK;
}

}  // extern "C"
