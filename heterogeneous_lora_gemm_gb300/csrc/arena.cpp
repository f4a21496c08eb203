#include "arena.h"

#include "../../include/mlora.h"

namespace mlora {

int Arena::alloc(int id, int n) {
    if (n <= 0 || where_.count(id)) return -1;
    const int size = round8(n);
    int cursor = 0;
    bool in_gap = false;
    for (const auto& kv : blocks_) {
        if (kv.first - cursor >= size) {   // hole before this block fits
            in_gap = true;
            break;
        }
        cursor = kv.first + kv.second.second;
    }
    if (!in_gap && units_ - cursor < size) return -1;   // tail hole too small
    blocks_[cursor] = {id, size};
    where_[id] = cursor;
    used_ += size;
    return cursor;
}

bool Arena::release(int id) {
    auto it = where_.find(id);
    if (it == where_.end()) return false;
    auto b = blocks_.find(it->second);
    used_ -= b->second.second;
    blocks_.erase(b);
    where_.erase(it);
    return true;
}

bool Arena::rename(int from, int to) {
    auto it = where_.find(from);
    if (it == where_.end() || where_.count(to)) return false;
    const int off = it->second;
    blocks_[off].first = to;
    where_.erase(it);
    where_[to] = off;
    return true;
}

int Arena::offset_of(int id) const {
    auto it = where_.find(id);
    return it == where_.end() ? -1 : it->second;
}

int Arena::largest_hole() const {
    int cursor = 0, best = 0;
    for (const auto& kv : blocks_) {
        if (kv.first - cursor > best) best = kv.first - cursor;
        cursor = kv.first + kv.second.second;
    }
    if (units_ - cursor > best) best = units_ - cursor;
    return best;
}

std::vector<ArenaMove> Arena::compact() {
    std::vector<ArenaMove> moves;
    std::map<int, std::pair<int, int>> packed;
    int cursor = 0;
    for (const auto& kv : blocks_) {
        const int id = kv.second.first, size = kv.second.second;
        if (kv.first != cursor) moves.push_back({id, kv.first, cursor, size});
        packed[cursor] = {id, size};
        where_[id] = cursor;
        cursor += size;
    }
    blocks_.swap(packed);
    return moves;
}

}  // namespace mlora

// ---- host-only C view for tests of the placement logic ----
struct mlora_arena {
    mlora::Arena a;
    explicit mlora_arena(int units) : a(units) {}
};

extern "C" {

mlora_arena_t mlora_arena_new(int units) {
    if (units < 0) return nullptr;
    return new mlora_arena(units);
}

void mlora_arena_delete(mlora_arena_t arena) { delete arena; }

int mlora_arena_alloc(mlora_arena_t arena, int id, int n) {
    return arena ? arena->a.alloc(id, n) : -1;
}

int mlora_arena_free(mlora_arena_t arena, int id) {
    return (arena && arena->a.release(id)) ? 0 : -1;
}

int mlora_arena_rename(mlora_arena_t arena, int from, int to) {
    return (arena && arena->a.rename(from, to)) ? 0 : -1;
}

int mlora_arena_compact(mlora_arena_t arena, int32_t* moves, int cap) {
    if (!arena) return -1;
    auto mv = arena->a.compact();
    int n = 0;
    for (const auto& m : mv) {
        if (moves && n < cap) {
            moves[3 * n + 0] = m.id;
            moves[3 * n + 1] = m.from;
            moves[3 * n + 2] = m.to;
        }
        ++n;
    }
    return n;
}

int mlora_arena_used(mlora_arena_t arena) { return arena ? arena->a.used() : -1; }

int mlora_arena_largest_hole(mlora_arena_t arena) { return arena ? arena->a.largest_hole() : -1; }

}  // extern "C"
