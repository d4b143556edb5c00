// Host block pool: the PagePool of the PagedAttention article ("Aufmerksamkeit"
// feed, chatgpz.de, SECTION 2 "Pages + Block Table" and SECTION 3
// "Copy-on-Write"), as native code.
//
//  alloc   -> pops the head of a FIFO free list, refcount 1 (empty: OOM)
//  share   -> refcount + 1 on a live block
//  release -> refcount - 1; at zero the block goes to the tail of the free list
//  refcount/num_free/utilisation are read-only queries
// Blocks that are not live cannot be shared or released (the article's
// dictionary would silently go negative; here it is an error).
#pragma once
#include <cstdint>
#include <deque>
#include <mutex>
#include <vector>

namespace kvc {

class BlockPool {
   public:
    explicit BlockPool(int32_t total) : total_(total), ref_(static_cast<size_t>(total), 0) {
        for (int32_t i = 0; i < total; ++i) free_.push_back(i);
    }
    int32_t total() const { return total_; }

    // All methods below are called with the mutex held by the caller (see lock()).
    std::unique_lock<std::mutex> lock() { return std::unique_lock<std::mutex>(mu_); }

    bool live(int32_t b) const { return b >= 0 && b < total_ && ref_[static_cast<size_t>(b)] > 0; }
    int32_t refcount(int32_t b) const { return (b >= 0 && b < total_) ? ref_[static_cast<size_t>(b)] : 0; }
    int32_t num_free() const { return static_cast<int32_t>(free_.size()); }

    // returns -1 when the free list is empty
    int32_t alloc() {
        if (free_.empty()) return -1;
        const int32_t b = free_.front();
        free_.pop_front();
        ref_[static_cast<size_t>(b)] = 1;
        return b;
    }
    void share(int32_t b) { ++ref_[static_cast<size_t>(b)]; }
    void release(int32_t b) {
        if (--ref_[static_cast<size_t>(b)] == 0) free_.push_back(b);
    }

   private:
    int32_t total_;
    std::deque<int32_t> free_;
    std::vector<int32_t> ref_;
    std::mutex mu_;
};

}  // namespace kvc
