// packer.cpp -- host-side packing of samples into fixed-length windows and the
// assignment of windows to data-parallel ranks: the data step in front of the
// attention path.  Declared in include/vlc.h (vlc_pack, vlc_shard_packs).
//
// Packing ("Sequence Packing", llm-compass, section on binning): windows of
// `capacity` tokens; a sample occupies its length plus `extra` tokens (the
// BOS/EOS reserve of the "Packing document boundary" checklist).  Three rules:
//   first-fit decreasing  samples by size, largest first (ties: smaller index),
//                         each into the first open window with room;
//   first-fit             the same without the sort (Megatron's dp_balanced
//                         order, as "Long-context training: remove padding"
//                         describes it);
//   next-fit              streaming: the current window or a new one.
// A sample larger than a window is not cut: it opens a window of its own,
// which takes nothing else, and is counted as oversize.
//
// First fit is answered by a max-segment-tree over the windows' free room: the
// leftmost window whose room is at least s is found by one root-to-leaf walk,
// so n samples take O(n log W) for W windows.  Sizes are ordered by a counting
// sort (stable, descending) when they are small, else by a stable comparison
// sort.
//
// Sharding ("Sequence packing and variable-length attention", charlestar: equal
// token counts can hide unequal attention work, balance sum(L^2)): windows by
// cost, largest first (ties: smaller index), each to the rank with the least
// load so far (ties: lower rank).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/vlc.h"

namespace {

// Max-tree over window room (int32: room never exceeds the capacity); leaves
// past the open windows hold -1 so that they are never chosen (a new window is
// opened explicitly).  An update climbs only while the parent's maximum changes.
class RoomTree {
public:
    explicit RoomTree(int64_t leaves) {
        size_ = 1;
        while (size_ < leaves) size_ <<= 1;
        t_.assign(static_cast<size_t>(2 * size_), -1);
    }
    void set(int64_t leaf, int32_t room) {
        int64_t i = leaf + size_;
        t_[i] = room;
        for (i >>= 1; i >= 1; i >>= 1) {
            const int32_t m = std::max(t_[2 * i], t_[2 * i + 1]);
            if (t_[i] == m) break;
            t_[i] = m;
        }
    }
    int32_t get(int64_t leaf) const { return t_[leaf + size_]; }
    // leftmost leaf with room >= s, or -1
    int64_t first_fit(int32_t s) const {
        if (t_[1] < s) return -1;
        int64_t i = 1;
        while (i < size_) i = (t_[2 * i] >= s) ? 2 * i : 2 * i + 1;
        return i - size_;
    }
    int64_t leaves() const { return size_; }

private:
    int64_t size_;
    std::vector<int32_t> t_;
};

// Stable order of sample indices by size, largest first.
std::vector<int64_t> decreasing_order(const std::vector<int64_t>& size) {
    const int64_t n = static_cast<int64_t>(size.size());
    std::vector<int64_t> idx(static_cast<size_t>(n));
    int64_t mx = 0;
    for (int64_t s : size) mx = std::max(mx, s);
    if (mx <= (int64_t(1) << 22)) {   // counting sort over the size values
        std::vector<int64_t> start(static_cast<size_t>(mx + 2), 0);
        for (int64_t s : size) ++start[static_cast<size_t>(mx - s + 1)];
        for (int64_t v = 1; v <= mx + 1; ++v) start[static_cast<size_t>(v)] += start[static_cast<size_t>(v - 1)];
        for (int64_t i = 0; i < n; ++i) idx[static_cast<size_t>(start[static_cast<size_t>(mx - size[i])]++)] = i;
    } else {
        for (int64_t i = 0; i < n; ++i) idx[static_cast<size_t>(i)] = i;
        std::stable_sort(idx.begin(), idx.end(), [&](int64_t a, int64_t b) { return size[a] > size[b]; });
    }
    return idx;
}

}  // namespace

extern "C" {

int vlc_pack(const int32_t* lengths, int64_t n, int32_t capacity, int32_t extra, int mode, int32_t* bin_of,
             int64_t* order, int64_t* bin_start, int64_t* nbins_out, int64_t* oversize_out) {
    if (lengths == nullptr || bin_of == nullptr || order == nullptr || bin_start == nullptr ||
        nbins_out == nullptr || n < 1 || capacity < 1 || extra < 0)
        return VLC_ERR_ARG;
    if (mode != VLC_PACK_FFD && mode != VLC_PACK_FIRST_FIT && mode != VLC_PACK_NEXT_FIT) return VLC_ERR_ARG;
    if (n > (int64_t(1) << 31) - 1) return VLC_ERR_UNSUPPORTED;   // window ids are int32
    std::vector<int64_t> size(static_cast<size_t>(n));
    int64_t fitting = 0, oversize = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (lengths[i] < 1) return VLC_ERR_ARG;
        size[static_cast<size_t>(i)] = static_cast<int64_t>(lengths[i]) + extra;
        if (size[static_cast<size_t>(i)] > capacity) ++oversize;
        else fitting += size[static_cast<size_t>(i)];
    }
    // first fit leaves at most one window at most half full, so the fitting samples use
    // fewer than 2 * fitting / capacity + 1 windows (and never more than there are samples)
    const int64_t bound = std::min<int64_t>(n, 2 * (fitting / capacity) + 2 + oversize);

    std::vector<int64_t> seq;   // placement sequence
    if (mode == VLC_PACK_FFD) {
        seq = decreasing_order(size);
    } else {
        seq.resize(static_cast<size_t>(n));
        for (int64_t i = 0; i < n; ++i) seq[static_cast<size_t>(i)] = i;
    }
    int64_t nbins = 0;
    if (mode == VLC_PACK_NEXT_FIT) {
        int64_t room = -1;
        for (int64_t i : seq) {
            const int64_t s = size[static_cast<size_t>(i)];
            if (s > capacity || s > room) {   // a new window (an oversize sample fills it alone)
                room = s > capacity ? 0 : capacity - s;
                bin_of[i] = static_cast<int32_t>(nbins++);
            } else {
                room -= s;
                bin_of[i] = static_cast<int32_t>(nbins - 1);
            }
        }
    } else {
        RoomTree tree(bound);
        for (int64_t i : seq) {
            const int64_t s = size[static_cast<size_t>(i)];
            const int64_t b = s > capacity ? -1 : tree.first_fit(static_cast<int32_t>(s));
            if (b < 0) {
                if (nbins >= tree.leaves()) return VLC_ERR_UNSUPPORTED;   // cannot happen (bound above)
                tree.set(nbins, s > capacity ? 0 : static_cast<int32_t>(capacity - s));
                bin_of[i] = static_cast<int32_t>(nbins++);
            } else {
                tree.set(b, tree.get(b) - static_cast<int32_t>(s));
                bin_of[i] = static_cast<int32_t>(b);
            }
        }
    }
    // group by window, each window's samples in placement order
    std::vector<int64_t> fill(static_cast<size_t>(nbins) + 1, 0);
    for (int64_t i = 0; i < n; ++i) ++fill[static_cast<size_t>(bin_of[i]) + 1];
    for (int64_t b = 0; b < nbins; ++b) fill[static_cast<size_t>(b + 1)] += fill[static_cast<size_t>(b)];
    std::memcpy(bin_start, fill.data(), sizeof(int64_t) * static_cast<size_t>(nbins + 1));
    for (int64_t i : seq) order[fill[static_cast<size_t>(bin_of[i])]++] = i;
    *nbins_out = nbins;
    if (oversize_out != nullptr) *oversize_out = oversize;
    return VLC_OK;
}

int vlc_shard_packs(const int32_t* lengths, const int64_t* order, const int64_t* bin_start, int64_t nbins,
                    int32_t ranks, int cost_kind, int32_t* rank_of_bin, int64_t* rank_load) {
    if (lengths == nullptr || order == nullptr || bin_start == nullptr || rank_of_bin == nullptr ||
        rank_load == nullptr || nbins < 1 || ranks < 1)
        return VLC_ERR_ARG;
    if (cost_kind != VLC_COST_TOKENS && cost_kind != VLC_COST_SUMSQ) return VLC_ERR_ARG;
    if (bin_start[0] != 0) return VLC_ERR_ARG;
    std::vector<int64_t> cost(static_cast<size_t>(nbins), 0);
    for (int64_t b = 0; b < nbins; ++b) {
        if (bin_start[b + 1] < bin_start[b]) return VLC_ERR_ARG;
        int64_t c = 0;
        for (int64_t k = bin_start[b]; k < bin_start[b + 1]; ++k) {
            const int64_t L = lengths[order[k]];
            if (L < 1) return VLC_ERR_ARG;
            const int64_t term = cost_kind == VLC_COST_SUMSQ ? L * L : L;
            if (__builtin_add_overflow(c, term, &c)) return VLC_ERR_UNSUPPORTED;
        }
        cost[static_cast<size_t>(b)] = c;
    }
    std::vector<int64_t> idx(static_cast<size_t>(nbins));
    for (int64_t b = 0; b < nbins; ++b) idx[static_cast<size_t>(b)] = b;
    std::stable_sort(idx.begin(), idx.end(), [&](int64_t a, int64_t b) { return cost[a] > cost[b]; });
    // min-heap of (load, rank): the least loaded rank, the lower rank on ties
    using Item = std::pair<int64_t, int32_t>;
    std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
    for (int32_t r = 0; r < ranks; ++r) {
        heap.emplace(0, r);
        rank_load[r] = 0;
    }
    for (int64_t b : idx) {
        Item top = heap.top();
        heap.pop();
        if (__builtin_add_overflow(top.first, cost[static_cast<size_t>(b)], &top.first)) return VLC_ERR_UNSUPPORTED;
        rank_of_bin[b] = top.second;
        rank_load[top.second] = top.first;
        heap.push(top);
    }
    return VLC_OK;
}

}  // extern "C"
