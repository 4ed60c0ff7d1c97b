// Host block allocator: free list + reference counts + copy-on-write.
//
// Policy ("Efficient Memory Management for LLM Serving with PagedAttention",
// azimuth.plus summary, sections "vLLM" and "Memory sharing"; CSDN tutorial
// "PagedAttention实战" §2.2 BlockManager, §3.1 append_kv, §5.1 clone_sequence):
//   - all blocks exist up front; the free list is a stack whose top is its last
//     element (the tutorial pops from the end of a Python list);
//   - allocating sets refcount 1, forking adds 1 to every shared block, freeing
//     subtracts 1 and pushes a block back when it reaches 0;
//   - a token lands at logical block pos / B, offset pos % B; writing into a block
//     that other sequences still reference copies that block first.
// Host memory only; every failure leaves the state unchanged.
#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pa_alloc {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;            // top = back()
    std::vector<int32_t> refs;
    int num_host_blocks = 0;                    // swap space in host memory
    std::vector<int32_t> host_free;             // top = back()
    std::vector<int32_t> host_refs;
    struct Seq {
        bool live = false;
        bool swapped = false;                   // blocks are host-pool ids
        int64_t len = 0;
        std::vector<int32_t> blocks;
    };
    std::vector<Seq> seqs;                      // index = sequence id
};

namespace {

bool live(const pa_alloc *a, int seq)
{
    return a && seq >= 0 && seq < (int)a->seqs.size() && a->seqs[seq].live;
}

bool resident(const pa_alloc *a, int seq) { return live(a, seq) && !a->seqs[seq].swapped; }

// Move every reference of seqs[0..n) from one pool to the other (swap out: device
// -> host; swap in: host -> device).  Each distinct source block, met in sequence
// order then table order, takes the top of the target pool's free stack; pairs get
// (source, target) in that order.  Source blocks whose count reaches zero go to the
// end of their free stack in the order the references are released.  All or
// nothing: the checks come first.
pa_status move_seqs(pa_alloc *a, const int *seqs, int n, bool out, int32_t *pairs, int cap,
                    int *num_pairs)
{
    if (!a || n < 0 || (n > 0 && !seqs) || !num_pairs || cap < 0 || (cap > 0 && !pairs))
        return PA_ERR_INVALID;
    std::vector<int32_t> &src_refs = out ? a->refs : a->host_refs;
    std::vector<int32_t> &dst_refs = out ? a->host_refs : a->refs;
    std::vector<int32_t> &src_free = out ? a->free_stack : a->host_free;
    std::vector<int32_t> &dst_free = out ? a->host_free : a->free_stack;
    std::unordered_map<int32_t, int32_t> target;
    std::vector<int32_t> order;
    try {
        for (int i = 0; i < n; ++i) {
            const int q = seqs[i];
            if (!live(a, q) || a->seqs[q].swapped != !out)
                return PA_ERR_INVALID;
            for (int k = 0; k < i; ++k)
                if (seqs[k] == q)
                    return PA_ERR_INVALID;
            for (int32_t b : a->seqs[q].blocks)
                if (target.emplace(b, -1).second)
                    order.push_back(b);
        }
        src_free.reserve(src_refs.size());
    } catch (...) {
        return PA_ERR_OOM;
    }
    *num_pairs = (int)order.size();
    if (order.size() > dst_free.size())
        return PA_ERR_OOM;
    if ((size_t)cap < order.size())
        return PA_ERR_INVALID;
    for (size_t i = 0; i < order.size(); ++i) {
        const int32_t t = dst_free.back();
        dst_free.pop_back();
        dst_refs[t] = 0;
        target[order[i]] = t;
        pairs[2 * i] = order[i];
        pairs[2 * i + 1] = t;
    }
    for (int i = 0; i < n; ++i) {
        pa_alloc::Seq &sq = a->seqs[seqs[i]];
        for (int32_t &b : sq.blocks) {
            const int32_t t = target[b];
            dst_refs[t] += 1;
            if (--src_refs[b] == 0)
                src_free.push_back(b);
            b = t;
        }
        sq.swapped = out;
    }
    return PA_OK;
}

// One append; `stage` receives the copy pair.  No state changes on PA_ERR_OOM.
pa_status append_one(pa_alloc *a, int seq, int64_t *slot, int32_t *src, int32_t *dst)
{
    pa_alloc::Seq &s = a->seqs[seq];
    const int64_t pos = s.len;
    const size_t logical = (size_t)(pos / a->block_size);
    const int offset = (int)(pos % a->block_size);
    *src = -1;
    *dst = -1;
    if (logical == s.blocks.size()) {
        if (a->free_stack.empty())
            return PA_ERR_OOM;
        const int32_t b = a->free_stack.back();
        a->free_stack.pop_back();
        a->refs[b] = 1;
        s.blocks.push_back(b);
    } else {
        const int32_t old = s.blocks[logical];
        if (a->refs[old] > 1) {
            if (a->free_stack.empty())
                return PA_ERR_OOM;
            const int32_t b = a->free_stack.back();
            a->free_stack.pop_back();
            a->refs[b] = 1;
            a->refs[old] -= 1;
            s.blocks[logical] = b;
            *src = old;
            *dst = b;
        }
    }
    s.len = pos + 1;
    *slot = (int64_t)s.blocks[logical] * a->block_size + offset;
    return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_alloc_create(pa_alloc **out, int num_blocks, int block_size, const int32_t *free_order)
{
    if (!out || num_blocks <= 0 || block_size <= 0)
        return PA_ERR_INVALID;
    *out = nullptr;
    pa_alloc *a = new (std::nothrow) pa_alloc;
    if (!a)
        return PA_ERR_OOM;
    try {
        a->num_blocks = num_blocks;
        a->block_size = block_size;
        a->refs.assign(num_blocks, 0);
        a->free_stack.resize(num_blocks);
        if (free_order) {
            std::vector<char> seen(num_blocks, 0);
            for (int i = 0; i < num_blocks; ++i) {
                const int32_t b = free_order[i];
                if (b < 0 || b >= num_blocks || seen[b]) {
                    delete a;
                    return PA_ERR_INVALID;
                }
                seen[b] = 1;
                a->free_stack[i] = b;
            }
        } else {
            for (int i = 0; i < num_blocks; ++i)
                a->free_stack[i] = i;
        }
    } catch (...) {
        delete a;
        return PA_ERR_OOM;
    }
    *out = a;
    return PA_OK;
}

void pa_alloc_destroy(pa_alloc *a) { delete a; }

pa_status pa_alloc_new_seq(pa_alloc *a, int *seq_id)
{
    if (!a || !seq_id)
        return PA_ERR_INVALID;
    try {
        a->seqs.emplace_back();
    } catch (...) {
        return PA_ERR_OOM;
    }
    a->seqs.back().live = true;
    *seq_id = (int)a->seqs.size() - 1;
    return PA_OK;
}

pa_status pa_alloc_fork(pa_alloc *a, int parent, int *child)
{
    if (!resident(a, parent) || !child)
        return PA_ERR_INVALID;
    try {
        pa_alloc::Seq c;
        c.live = true;
        c.len = a->seqs[parent].len;
        c.blocks = a->seqs[parent].blocks;
        a->seqs.push_back(std::move(c));
    } catch (...) {
        return PA_ERR_OOM;
    }
    for (int32_t b : a->seqs.back().blocks)
        a->refs[b] += 1;
    *child = (int)a->seqs.size() - 1;
    return PA_OK;
}

pa_status pa_alloc_append(pa_alloc *a, int seq, int64_t *slot, int32_t *cow_src, int32_t *cow_dst)
{
    if (!resident(a, seq) || !slot)
        return PA_ERR_INVALID;
    int32_t s = -1, d = -1;
    try {
        a->seqs[seq].blocks.reserve(a->seqs[seq].blocks.size() + 1);
    } catch (...) {
        return PA_ERR_OOM;
    }
    const pa_status st = append_one(a, seq, slot, &s, &d);
    if (cow_src)
        *cow_src = s;
    if (cow_dst)
        *cow_dst = d;
    return st;
}

pa_status pa_alloc_append_n(pa_alloc *a, int seq, int n, int64_t *slots, int32_t *cow_pairs,
                            int *num_cow, int *done)
{
    if (!resident(a, seq) || n < 0 || (n > 0 && !slots) || !num_cow)
        return PA_ERR_INVALID;
    *num_cow = 0;
    if (done)
        *done = 0;
    for (int i = 0; i < n; ++i) {
        int32_t s, d;
        try {
            a->seqs[seq].blocks.reserve(a->seqs[seq].blocks.size() + 1);
        } catch (...) {
            return PA_ERR_OOM;
        }
        const pa_status st = append_one(a, seq, &slots[i], &s, &d);
        if (st != PA_OK)
            return st;
        if (s >= 0 && cow_pairs) {
            cow_pairs[2 * *num_cow] = s;
            cow_pairs[2 * *num_cow + 1] = d;
        }
        if (s >= 0)
            *num_cow += 1;
        if (done)
            *done = i + 1;
    }
    return PA_OK;
}

pa_status pa_alloc_free_seq(pa_alloc *a, int seq)
{
    if (!live(a, seq))
        return PA_ERR_INVALID;
    pa_alloc::Seq &s = a->seqs[seq];
    std::vector<int32_t> &refs = s.swapped ? a->host_refs : a->refs;
    std::vector<int32_t> &stack = s.swapped ? a->host_free : a->free_stack;
    // a free stack never exceeds its pool's size, so reserve up front
    try {
        stack.reserve(refs.size());
    } catch (...) {
        return PA_ERR_OOM;
    }
    for (int32_t b : s.blocks) {
        refs[b] -= 1;
        if (refs[b] == 0)
            stack.push_back(b);
    }
    s.blocks.clear();
    s.blocks.shrink_to_fit();
    s.len = 0;
    s.live = false;
    s.swapped = false;
    return PA_OK;
}

pa_status pa_alloc_block_table(const pa_alloc *a, int seq, int32_t *out, int cap, int *n)
{
    if (!live(a, seq) || !n || cap < 0 || (cap > 0 && !out))
        return PA_ERR_INVALID;
    const std::vector<int32_t> &b = a->seqs[seq].blocks;
    *n = (int)b.size();
    std::copy(b.begin(), b.begin() + std::min<size_t>(b.size(), (size_t)cap), out);
    return PA_OK;
}

pa_status pa_alloc_seq_len(const pa_alloc *a, int seq, int *len)
{
    if (!live(a, seq) || !len)
        return PA_ERR_INVALID;
    *len = (int)a->seqs[seq].len;
    return PA_OK;
}

int pa_alloc_refcount(const pa_alloc *a, int block)
{
    if (!a || block < 0 || block >= a->num_blocks)
        return -1;
    return a->refs[block];
}

int pa_alloc_num_free(const pa_alloc *a) { return a ? (int)a->free_stack.size() : -1; }

pa_status pa_alloc_free_list(const pa_alloc *a, int32_t *out, int cap, int *n)
{
    if (!a || !n || cap < 0 || (cap > 0 && !out))
        return PA_ERR_INVALID;
    *n = (int)a->free_stack.size();
    std::copy(a->free_stack.begin(),
              a->free_stack.begin() + std::min<size_t>(a->free_stack.size(), (size_t)cap), out);
    return PA_OK;
}

pa_status pa_alloc_usage_stats(const pa_alloc *a, pa_alloc_usage *out)
{
    if (!a || !out)
        return PA_ERR_INVALID;
    pa_alloc_usage u = {};
    // rows of each device block that hold a token of some resident sequence: rows
    // fill from 0 upward, so it is the largest count any holder has in it
    std::vector<int32_t> rows;
    try {
        rows.assign(a->num_blocks, 0);
    } catch (...) {
        return PA_ERR_OOM;
    }
    for (const pa_alloc::Seq &q : a->seqs) {
        if (!q.live)
            continue;
        if (q.swapped) {
            u.swapped_seqs += 1;
            continue;
        }
        u.resident_seqs += 1;
        u.logical_blocks += (int64_t)q.blocks.size();
        for (size_t j = 0; j < q.blocks.size(); ++j) {
            const int64_t r = std::min<int64_t>(a->block_size, q.len - (int64_t)j * a->block_size);
            rows[q.blocks[j]] = std::max<int32_t>(rows[q.blocks[j]], (int32_t)r);
        }
    }
    for (int b = 0; b < a->num_blocks; ++b) {
        if (a->refs[b] > 0) {
            u.used_blocks += 1;
            u.tokens += rows[b];
        }
    }
    u.token_slots = u.used_blocks * a->block_size;
    *out = u;
    return PA_OK;
}

pa_status pa_alloc_set_host_pool(pa_alloc *a, int num_host_blocks)
{
    if (!a || num_host_blocks < 0)
        return PA_ERR_INVALID;
    for (const pa_alloc::Seq &q : a->seqs)
        if (q.live && q.swapped)
            return PA_ERR_INVALID;
    try {
        a->host_refs.assign(num_host_blocks, 0);
        a->host_free.resize(num_host_blocks);
    } catch (...) {
        return PA_ERR_OOM;
    }
    for (int i = 0; i < num_host_blocks; ++i)
        a->host_free[i] = i;
    a->num_host_blocks = num_host_blocks;
    return PA_OK;
}

pa_status pa_alloc_swap_out(pa_alloc *a, const int *seqs, int n, int32_t *pairs, int cap,
                            int *num_pairs)
{
    return move_seqs(a, seqs, n, true, pairs, cap, num_pairs);
}

pa_status pa_alloc_swap_in(pa_alloc *a, const int *seqs, int n, int32_t *pairs, int cap,
                           int *num_pairs)
{
    return move_seqs(a, seqs, n, false, pairs, cap, num_pairs);
}

int pa_alloc_is_swapped(const pa_alloc *a, int seq)
{
    return live(a, seq) ? (a->seqs[seq].swapped ? 1 : 0) : -1;
}

int pa_alloc_host_refcount(const pa_alloc *a, int block)
{
    if (!a || block < 0 || block >= a->num_host_blocks)
        return -1;
    return a->host_refs[block];
}

int pa_alloc_num_free_host(const pa_alloc *a) { return a ? (int)a->host_free.size() : -1; }

pa_status pa_alloc_host_free_list(const pa_alloc *a, int32_t *out, int cap, int *n)
{
    if (!a || !n || cap < 0 || (cap > 0 && !out))
        return PA_ERR_INVALID;
    *n = (int)a->host_free.size();
    std::copy(a->host_free.begin(),
              a->host_free.begin() + std::min<size_t>(a->host_free.size(), (size_t)cap), out);
    return PA_OK;
}

}  // extern "C"

// Shared-prefix groups for pa_decode_shared, from the block tables alone: a group
// is a maximal run of consecutive batch rows whose first entries name the same
// physical block; it shares the leading entries common to all its rows, capped so
// that every member's newest token stays outside the shared part.
pa_status pa_share_groups(const int32_t *block_tables, int num_seqs, int max_blocks_per_seq,
                          const int32_t *context_lens, int block_size, int min_shared_blocks,
                          int32_t *share)
{
    if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0 || min_shared_blocks < 1)
        return PA_ERR_INVALID;
    if (num_seqs > 0 && (!block_tables || !context_lens || !share || max_blocks_per_seq == 0))
        return PA_ERR_INVALID;
    const size_t W = (size_t)max_blocks_per_seq;
    auto cap = [&](int s) {     // blocks of s that hold no newest token: floor((T-1)/B)
        const int T = context_lens[s];
        return T <= 0 ? 0 : std::min((T - 1) / block_size, max_blocks_per_seq);
    };
    int g = 0;
    while (g < num_seqs) {
        const int32_t *row0 = block_tables + (size_t)g * W;
        int e = g + 1;
        while (e < num_seqs && row0[0] >= 0 && block_tables[(size_t)e * W] == row0[0])
            ++e;
        int P = cap(g);
        for (int m = g + 1; m < e; ++m) {
            const int32_t *row = block_tables + (size_t)m * W;
            int j = 0;
            const int lim = std::min(P, cap(m));
            while (j < lim && row[j] == row0[j] && row[j] >= 0)
                ++j;
            P = j;
        }
        const bool ok = e - g >= 2 && P >= min_shared_blocks;
        for (int m = g; m < e; ++m) {
            share[2 * m] = ok ? g : -1;
            share[2 * m + 1] = ok ? P : 0;
        }
        g = e;
    }
    return PA_OK;
}
