// Rank-unit arena allocator of the adapter pool (host side, no CUDA).
//
// The pool keeps every resident adapter in one device arena measured in rank
// units: an adapter of rank r holds roundup(r, 8) consecutive units, i.e. its
// Down rows and its Up block sit at unit offset u in the two arena halves.
// Blocks start at multiples of 8 units.  Placement is first fit; when no hole is
// large enough but the total free space is, the pool compacts (slides live blocks
// toward offset 0 in order) and retries, so the rank budget is honoured exactly
// (no fragmentation loss).  This replaces a max_slots x max_rank slot grid (the
// wiblog failure mode where one high-rank adapter inflates every slot).
#pragma once
#include <cstdint>
#include <map>
#include <unordered_map>
#include <vector>

namespace mlora {

struct ArenaMove {
    int id, from, to, size;
};

class Arena {
public:
    explicit Arena(int units) : units_(units) {}

    static int round8(int n) { return (n + 7) & ~7; }

    int units() const { return units_; }
    int used() const { return used_; }
    int free_units() const { return units_ - used_; }

    // First-fit placement of round8(n) units for `id`; -1 if no hole fits.
    int alloc(int id, int n);
    // Releases the block of `id`; false if `id` holds none.
    bool release(int id);
    // Gives the block of `from` to `to` (which holds none), in place; false otherwise.
    bool rename(int from, int to);
    // Unit offset of `id`'s block, or -1.
    int offset_of(int id) const;
    int largest_hole() const;
    // Slides live blocks toward 0 keeping their order; returns the moves made.
    std::vector<ArenaMove> compact();

private:
    int units_;
    int used_ = 0;
    std::map<int, std::pair<int, int>> blocks_;   // offset -> (id, size)
    std::unordered_map<int, int> where_;          // id -> offset
};

}  // namespace mlora
