// C ABI of libmlora.so: the adapter pool (device-resident slot pool with a
// rank-packed arena) and the entry points declared in include/mlora.h.
//
// Host side only: argument checks, the arena allocator, copies into the arena,
// and launches.  Every step of the forward and of the merge runs in this
// library's CUDA kernels; there is no CPU fallback.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdarg>
#include <map>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/mlora.h"
#include "arena.h"
#include "internal.h"
#include "tc.h"

using namespace mlora;

namespace {

thread_local std::string g_last_error;

mlora_status fail(mlora_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

mlora_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MLORA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define CU_TRY(expr)                                              \
    do {                                                          \
        cudaError_t e_ = (expr);                                  \
        if (e_ != cudaSuccess) return cuda_fail(e_, #expr);       \
    } while (0)

// Makes the pool's device current for the scope of one call and restores the caller's.
struct DeviceGuard {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

struct SlotHost {
    int rank = 0;
    int rpad = 0;
    float scale = 0.f;
    int unit = -1;
    uint64_t version = 0;
    // per chunk: output rows its Up columns reach (modules of a fused projection);
    // empty for an adapter of the whole layer
    std::vector<std::pair<int, int>> chunk_rows;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// bf16 <-> fp32 on the host: bf16 is the upper half of an fp32; rounding to nearest,
// ties to even, on the dropped lower half (inputs here are finite)
float bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}
uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

}  // namespace

void mlora::set_last_error(const std::string& msg) { g_last_error = msg; }

struct mlora_pool {
    int device = 0;
    int max_slots = 0, max_rank = 0, din = 0, dout = 0, max_tokens = 0;
    mlora_dtype dtype = MLORA_BF16;
    size_t esize = 2;
    int units = 0;
    Arena arena{0};
    std::vector<SlotHost> slots;
    int loaded = 0;

    // device memory
    char* arena_base = nullptr;      // Down half [units x din], then Up half [units x dout]
    char* arena_down = nullptr;
    char* arena_up = nullptr;
    size_t arena_bytes = 0;
    char* table_base = nullptr;      // two table sets, each the slot table then the chunk table
    size_t slots_bytes = 0;          // the slot table's share of a set (the chunk table follows)
    SlotRec* set_slots[2] = {nullptr, nullptr};
    ChunkRec* set_chunks[2] = {nullptr, nullptr};
    int cur = 0;                     // the set that forwards enqueued now read
    cudaEvent_t set_retired[2] = {nullptr, nullptr};   // set s's readers done (recorded when it stopped being current)
    bool set_retired_pending[2] = {false, false};
    SlotRec* d_slots = nullptr;      // = set_slots[cur]
    ChunkRec* d_chunks = nullptr;    // = set_chunks[cur]: chunks of the loaded slots, in arena order
    int n_chunks = 0;
    int tile_span = 0;               // largest arena span of 8 consecutive chunks of the table
    int run_stride = 0;              // most common arena stride of 4-chunk K-extension units (0: none)
    TcArenaMaps maps{};              // TMA descriptors of the whole arena (bf16 pools)
    size_t table_bytes = 0;
    char* ws_base = nullptr;
    size_t ws_bytes = 0;
    Workspace ws{};
    uint32_t* row_max = nullptr;     // quantized merge: per-row max word (zero between calls)
    PoolDims dims{};

    cudaStream_t copy_stream = nullptr;
    cudaEvent_t last_reader = nullptr;
    bool reader_pending = false;
    bool captured = false;           // a forward or merge was captured into a graph

    unsigned long long* prof_stamps = nullptr;   // caller's profiling record buffer (NULL = off)
    int prof_cap = 0;
    int last_T = 0;                  // rows of the last forward that built segments

    // Host (cold) tier (M031 §06): adapters in pinned host memory, already in the
    // arena's layout, copied into a slot on demand by mlora_prefetch.
    struct HostAdapter {
        char* down = nullptr;        // [rpad x din]
        char* up = nullptr;          // [rpad / 8 blocks][dout][8]
        int rank = 0, rpad = 0;
        float scale = 0.f;
        cudaEvent_t busy = nullptr;  // recorded after the last copy out of it
        bool busy_pending = false;
    };
    std::map<int, HostAdapter> cold;
    // Blocks of adapters evicted by a prefetch: kept out of the allocator (renamed to
    // a quarantine id) until `free_at`, recorded once their last reader finished.
    struct Quarantine {
        int id;
        cudaEvent_t free_at;
    };
    std::vector<Quarantine> quarantine;
    int next_qid = 0;
    // Pinned staging of the slot and chunk tables for their asynchronous updates: a
    // ring, each entry reused once the copy out of it is done.
    struct TableStage {
        char* buf = nullptr;
        cudaEvent_t done = nullptr;
        bool pending = false;
    };
    std::vector<TableStage> stages;
    int stage_next = 0;
    cudaEvent_t tables_ready = nullptr;   // the last asynchronous table update has landed
};

namespace {

mlora_status wait_readers(mlora_pool* p) {
    if (p->captured) {
        // graph replays of captured calls are invisible to the pool: wait for the device
        CU_TRY(cudaDeviceSynchronize());
        p->reader_pending = false;
        return MLORA_OK;
    }
    if (p->reader_pending) {
        CU_TRY(cudaEventSynchronize(p->last_reader));
        p->reader_pending = false;
    }
    return MLORA_OK;
}

mlora_status push_slot(mlora_pool* p, int slot) {
    const SlotHost& h = p->slots[slot];
    SlotRec rec{h.rank, h.rpad, h.scale, h.unit < 0 ? 0 : h.unit, 0};   // chunk0: set by push_chunks
    CU_TRY(cudaMemcpyAsync(p->d_slots + slot, &rec, sizeof rec, cudaMemcpyHostToDevice, p->copy_stream));
    // the staging object above lives on this stack frame: finish before returning
    CU_TRY(cudaStreamSynchronize(p->copy_stream));
    return MLORA_OK;
}

// Rewrites the chunk table of the loaded slots after a load, unload or move (no
// forward reads it meanwhile: every caller waited for the pool's last reader).
// The table is in arena order within each module (output row range) of a fused
// projection, modules in row order: 8 consecutive chunks (one row tile of the
// tensor-core shrink) usually lie in one window of at most 128 arena rows, and the
// K-extension units (4 consecutive chunks) of a row tile hold chunks of its own module.
mlora_status build_chunks(mlora_pool* p, std::vector<ChunkRec>& host) {
    host.clear();
    for (int s = 0; s < p->max_slots; ++s) {
        const SlotHost& h = p->slots[s];
        if (h.rank <= 0) continue;
        for (int j = 0; j * CHUNK < h.rank; ++j) {
            const int kv = h.rank - j * CHUNK;
            const bool mod = j < (int)h.chunk_rows.size();
            host.push_back(ChunkRec{s, h.unit + j * CHUNK, kv < CHUNK ? kv : CHUNK, h.scale,
                                    mod ? h.chunk_rows[j].first : 0, mod ? h.chunk_rows[j].second : p->dout});
        }
    }
    std::sort(host.begin(), host.end(), [](const ChunkRec& x, const ChunkRec& y) {
        return x.row0 != y.row0 ? x.row0 < y.row0 : x.unit < y.unit;
    });
    if ((int)host.size() > p->dims.max_chunks)
        return fail(MLORA_ERR_CUDA, "chunk table overflow: %zu > %d", host.size(), p->dims.max_chunks);
    p->n_chunks = (int)host.size();
    p->tile_span = 0;
    for (size_t t0 = 0; t0 < host.size(); t0 += 8) {
        // a window starts at the tile's first chunk: units must not decrease within the
        // tile (they may where one module's chunks end and the next module's begin)
        const size_t t1 = (t0 + 8 < host.size() ? t0 + 8 : host.size()) - 1;
        int span = host[t1].unit + CHUNK - host[t0].unit;
        for (size_t c = t0 + 1; c <= t1; ++c)
            if (host[c].unit < host[c - 1].unit) span = INT_MAX;
        if (span > p->tile_span) p->tile_span = span;
    }
    // K-extension units (4 consecutive chunks of the table) whose chunks lie at one
    // stride in the arena, within one module: the most common such stride lets a
    // projection load a unit's Up tiles in one box (e.g. the q chunks of tenants whose
    // slots each hold a q and a v adapter of one rank)
    std::map<int, int> votes;
    for (size_t u0 = 0; u0 + 4 <= host.size(); u0 += 4) {
        const int d = host[u0 + 1].unit - host[u0].unit;
        bool run = d >= CHUNK;
        for (size_t j = 1; j < 4 && run; ++j)
            run = host[u0 + j].unit - host[u0 + j - 1].unit == d && host[u0 + j].row0 == host[u0].row0 &&
                  host[u0 + j].row1 == host[u0].row1;
        if (run) ++votes[d];
    }
    p->run_stride = 0;
    int best = 0;
    for (const auto& v : votes)
        if (v.second > best) {
            best = v.second;
            p->run_stride = v.first;
        }
    return MLORA_OK;
}

// The slot table's records, each with the index of its slot's first chunk in `chunks`
// (the lowest; in a fused projection the slot's chunks of other modules come later).
void slot_records(const mlora_pool* p, const std::vector<ChunkRec>& chunks, SlotRec* out) {
    for (int s = 0; s < p->max_slots; ++s) {
        const SlotHost& h = p->slots[s];
        out[s] = SlotRec{h.rank, h.rpad, h.scale, h.unit < 0 ? 0 : h.unit, 0};
    }
    for (int c = (int)chunks.size() - 1; c >= 0; --c) out[chunks[c].slot].chunk0 = c;
}

mlora_status push_chunks(mlora_pool* p) {
    std::vector<ChunkRec> host;
    mlora_status st = build_chunks(p, host);
    if (st != MLORA_OK) return st;
    std::vector<SlotRec> recs((size_t)(p->max_slots > 0 ? p->max_slots : 1));
    slot_records(p, host, recs.data());
    if (p->max_slots > 0)
        CU_TRY(cudaMemcpyAsync(p->d_slots, recs.data(), sizeof(SlotRec) * (size_t)p->max_slots,
                               cudaMemcpyHostToDevice, p->copy_stream));
    if (!host.empty())
        CU_TRY(cudaMemcpyAsync(p->d_chunks, host.data(), sizeof(ChunkRec) * host.size(), cudaMemcpyHostToDevice,
                               p->copy_stream));
    // the staging vectors live on this stack frame: finish before returning
    CU_TRY(cudaStreamSynchronize(p->copy_stream));
    return MLORA_OK;
}

// Moves `size` units of both arena halves from unit `from` down to unit `to` (to < from),
// chunk by chunk so that no single copy overlaps itself.
mlora_status move_units(mlora_pool* p, int from, int to, int size) {
    const int shift = from - to;
    for (int off = 0; off < size; off += shift) {
        const int n = (size - off) < shift ? (size - off) : shift;
        const size_t drow = (size_t)p->din * p->esize, urow = (size_t)p->dout * p->esize;
        CU_TRY(cudaMemcpyAsync(p->arena_down + (size_t)(to + off) * drow, p->arena_down + (size_t)(from + off) * drow,
                               (size_t)n * drow, cudaMemcpyDeviceToDevice, p->copy_stream));
        CU_TRY(cudaMemcpyAsync(p->arena_up + (size_t)(to + off) * urow, p->arena_up + (size_t)(from + off) * urow,
                               (size_t)n * urow, cudaMemcpyDeviceToDevice, p->copy_stream));
    }
    return MLORA_OK;
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

constexpr int QUARANTINE_ID0 = 1 << 28;   // arena ids of quarantined blocks (slots are below)
constexpr int TABLE_STAGES = 4;

// Returns quarantined blocks whose last reader has finished to the allocator; with
// `wait`, waits for all of them first.
mlora_status reclaim(mlora_pool* p, bool wait) {
    std::vector<mlora_pool::Quarantine> keep;
    mlora_status st = MLORA_OK;
    for (const auto& q : p->quarantine) {
        cudaError_t e = cudaErrorNotReady;
        if (st == MLORA_OK) e = wait ? cudaEventSynchronize(q.free_at) : cudaEventQuery(q.free_at);
        if (e != cudaSuccess) {
            // not finished, or the query failed (the block stays out of the allocator)
            if (e != cudaErrorNotReady) st = cuda_fail(e, "quarantine event");
            keep.push_back(q);
            continue;
        }
        p->arena.release(q.id);
        cudaEventDestroy(q.free_at);
    }
    p->quarantine.swap(keep);   // only the blocks not returned above
    return st;
}

// Copies the host mirrors of the slot table and the chunk table into table set
// `set` on the copy stream, as one copy from a pinned staging entry laid out like
// the set, without waiting on the host (unless every entry of the ring is still in
// flight).  The caller has ordered the copy stream behind the set's readers.
mlora_status push_tables_async(mlora_pool* p, int set) {
    std::vector<ChunkRec> chunks;
    mlora_status st = build_chunks(p, chunks);
    if (st != MLORA_OK) return st;
    mlora_pool::TableStage& sg = p->stages[p->stage_next];
    p->stage_next = (p->stage_next + 1) % (int)p->stages.size();
    if (sg.pending) CU_TRY(cudaEventSynchronize(sg.done));
    SlotRec* recs = reinterpret_cast<SlotRec*>(sg.buf);
    slot_records(p, chunks, recs);
    ChunkRec* cr = reinterpret_cast<ChunkRec*>(sg.buf + p->slots_bytes);
    std::copy(chunks.begin(), chunks.end(), cr);
    CU_TRY(cudaMemcpyAsync(p->set_slots[set], sg.buf, p->slots_bytes + sizeof(ChunkRec) * chunks.size(),
                           cudaMemcpyHostToDevice, p->copy_stream));
    CU_TRY(cudaEventRecord(sg.done, p->copy_stream));
    sg.pending = true;
    return MLORA_OK;
}

// Records the pool's last-reader event after a forward/merge, or notes that the
// call went into a graph under capture (then later loads wait for the device).
mlora_status note_reader(mlora_pool* p, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CU_TRY(cudaStreamIsCapturing(st, &cs));
    if (cs != cudaStreamCaptureStatusNone) {
        p->captured = true;
        return MLORA_OK;
    }
    CU_TRY(cudaEventRecord(p->last_reader, st));
    p->reader_pending = true;
    return MLORA_OK;
}

}  // namespace

extern "C" {

const char* mlora_status_string(mlora_status s) {
    switch (s) {
        case MLORA_OK: return "ok";
        case MLORA_ERR_INVALID_ARG: return "invalid argument";
        case MLORA_ERR_BAD_SLOT: return "slot out of range";
        case MLORA_ERR_RANK: return "rank out of range";
        case MLORA_ERR_NOT_LOADED: return "slot holds no adapter";
        case MLORA_ERR_OOM: return "out of memory (rank budget or device)";
        case MLORA_ERR_CUDA: return "CUDA error";
        case MLORA_ERR_DEVICE_ROW: return "a row named an invalid or empty slot";
        case MLORA_ERR_UNSUPPORTED: return "unsupported shape";
        case MLORA_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait gave up";
    }
    return "unknown status";
}

const char* mlora_last_error(void) { return g_last_error.c_str(); }

mlora_status mlora_pool_create(int max_slots, int rank_budget, int max_rank, int din, int dout,
                               mlora_dtype dtype, int max_tokens, mlora_pool_t* out) {
    if (!out) return fail(MLORA_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (max_slots < 0 || max_slots > 4096) return fail(MLORA_ERR_INVALID_ARG, "max_slots %d not in [0, 4096]", max_slots);
    if (rank_budget < 0) return fail(MLORA_ERR_INVALID_ARG, "rank_budget %d < 0", rank_budget);
    if (max_rank < 1 || max_rank > 256) return fail(MLORA_ERR_INVALID_ARG, "max_rank %d not in [1, 256]", max_rank);
    if (din < 1 || dout < 1) return fail(MLORA_ERR_INVALID_ARG, "din %d / dout %d must be >= 1", din, dout);
    if (max_tokens < 1) return fail(MLORA_ERR_INVALID_ARG, "max_tokens %d < 1", max_tokens);
    if (dtype != MLORA_F32 && dtype != MLORA_BF16) return fail(MLORA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (dtype == MLORA_BF16 && din % 8 != 0)
        return fail(MLORA_ERR_UNSUPPORTED, "bf16 pools need din %% 8 == 0 (16-byte rows), got %d", din);
    if ((long long)rank_budget + 8 > (1ll << 30)) return fail(MLORA_ERR_INVALID_ARG, "rank_budget too large");

    mlora_pool* p = new mlora_pool();
    p->max_slots = max_slots;
    p->max_rank = max_rank;
    p->din = din;
    p->dout = dout;
    p->max_tokens = max_tokens;
    p->dtype = dtype;
    p->esize = dtype == MLORA_BF16 ? 2 : 4;
    p->units = Arena::round8(rank_budget);
    p->arena = Arena(p->units);
    p->slots.assign(max_slots, SlotHost{});

    auto bail = [&](mlora_status s) {
        mlora_pool_destroy(p);
        return s;
    };
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGetDevice"));

    // arena: Down half then Up half; unit offsets are multiples of 8, so every
    // Up block starts 16-byte aligned
    p->arena_bytes = align_up((size_t)p->units * din * p->esize, 256) + (size_t)p->units * dout * p->esize;
    if (p->arena_bytes > 0) {
        e = cudaMalloc((void**)&p->arena_base, p->arena_bytes);
        if (e != cudaSuccess) return bail(fail(MLORA_ERR_OOM, "arena of %zu bytes: %s", p->arena_bytes, cudaGetErrorString(e)));
        e = cudaMemset(p->arena_base, 0, p->arena_bytes);
        if (e != cudaSuccess) return bail(cuda_fail(e, "cudaMemset(arena)"));
    }
    p->arena_down = p->arena_base;
    p->arena_up = p->arena_base + align_up((size_t)p->units * din * p->esize, 256);

    // chunks of 16 rank columns: each slot's last chunk may be partial
    const int max_chunks = p->units / CHUNK + max_slots + 1;
    // slot table and chunk table
    // Two sets of (slot table, chunk table): forwards read the current one while a
    // prefetch writes the other, which then becomes current.
    const size_t slots_bytes = align_up(sizeof(SlotRec) * (size_t)(max_slots > 0 ? max_slots : 1), 128);
    const size_t set_bytes = slots_bytes + align_up(sizeof(ChunkRec) * (size_t)max_chunks, 128);
    p->slots_bytes = slots_bytes;
    p->table_bytes = 2 * set_bytes;
    e = cudaMalloc((void**)&p->table_base, p->table_bytes);
    if (e != cudaSuccess) return bail(fail(MLORA_ERR_OOM, "slot table: %s", cudaGetErrorString(e)));
    e = cudaMemset(p->table_base, 0, p->table_bytes);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaMemset(slot table)"));
    for (int k = 0; k < 2; ++k) {
        p->set_slots[k] = (SlotRec*)(p->table_base + k * set_bytes);
        p->set_chunks[k] = (ChunkRec*)(p->table_base + k * set_bytes + slots_bytes);
    }
    p->d_slots = p->set_slots[0];
    p->d_chunks = p->set_chunks[0];
    if (dtype == MLORA_BF16 && p->units > 0 &&
        !tc_encode_arena_maps(&p->maps, p->arena_down, p->arena_up, p->units, din, dout))
        return bail(fail(MLORA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the adapter arena"));

    // workspace
    PoolDims& d = p->dims;
    d.S = max_slots;
    d.din = din;
    d.dout = dout;
    d.max_rank = max_rank;
    d.max_tokens = max_tokens;
    d.max_chunks = max_chunks;
    d.tcap = (max_tokens + 15) / 16 * 16;
    const TcWorkspaceNeeds tcn = tc_workspace_needs(dtype == MLORA_BF16, d);
    size_t off = 0;
    auto carve = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    const size_t o_status = carve(4);
    const size_t o_counts = carve(sizeof(int32_t) * (size_t)(max_slots + 1));
    const size_t o_offsets = carve(sizeof(int32_t) * (size_t)(max_slots + 1));
    const size_t o_perm = carve(sizeof(int32_t) * (size_t)max_tokens);
    const size_t o_meta = carve(sizeof(int32_t) * 8);
    const size_t o_cslot = carve(sizeof(int32_t) * (size_t)d.max_chunks);
    const size_t o_cunit = carve(sizeof(int32_t) * (size_t)d.max_chunks);
    const size_t o_ckval = carve(sizeof(int32_t) * (size_t)d.max_chunks);
    const size_t o_v32 = carve(dtype == MLORA_F32 || tcn.need_v32 ? sizeof(float) * (size_t)max_tokens * max_rank : 0);
    const size_t o_vt = carve(dtype == MLORA_BF16 ? (size_t)d.max_chunks * d.tcap * CHUNK * 2 : 0);
    const size_t o_part = carve(tcn.partial_bytes);
    const size_t o_ctr = carve(tcn.counter_bytes);
    const size_t o_tmask = carve(tcn.tmask_bytes);
    const size_t o_rowmax = carve(sizeof(uint32_t) * (size_t)dout);
    p->ws_bytes = off;
    e = cudaMalloc((void**)&p->ws_base, p->ws_bytes);
    if (e != cudaSuccess) return bail(fail(MLORA_ERR_OOM, "workspace of %zu bytes: %s", p->ws_bytes, cudaGetErrorString(e)));
    e = cudaMemset(p->ws_base, 0, p->ws_bytes);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaMemset(workspace)"));
    Workspace& w = p->ws;
    w.status = (uint32_t*)(p->ws_base + o_status);
    w.counts = (int32_t*)(p->ws_base + o_counts);
    w.offsets = (int32_t*)(p->ws_base + o_offsets);
    w.perm = (int32_t*)(p->ws_base + o_perm);
    w.meta = (int32_t*)(p->ws_base + o_meta);
    w.chunk_slot = (int32_t*)(p->ws_base + o_cslot);
    w.chunk_unit = (int32_t*)(p->ws_base + o_cunit);
    w.chunk_kval = (int32_t*)(p->ws_base + o_ckval);
    w.v32 = (float*)(p->ws_base + o_v32);
    w.vt = (uint16_t*)(p->ws_base + o_vt);
    w.partials = (float*)(p->ws_base + o_part);
    w.tile_ctr = (int32_t*)(p->ws_base + o_ctr);
    w.chunks = p->d_chunks;
    w.tmask = (uint8_t*)(p->ws_base + o_tmask);
    p->row_max = (uint32_t*)(p->ws_base + o_rowmax);

    e = seg_init();
    if (e != cudaSuccess) return bail(cuda_fail(e, "seg_init"));
    e = tc_init();
    if (e != cudaSuccess) return bail(cuda_fail(e, "tc_init"));
    e = cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaStreamCreate"));
    e = cudaEventCreateWithFlags(&p->last_reader, cudaEventDisableTiming);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaEventCreate"));
    e = cudaEventCreateWithFlags(&p->tables_ready, cudaEventDisableTiming);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaEventCreate"));
    for (int k = 0; k < 2; ++k) {
        e = cudaEventCreateWithFlags(&p->set_retired[k], cudaEventDisableTiming);
        if (e != cudaSuccess) return bail(cuda_fail(e, "cudaEventCreate"));
    }
    p->stages.resize(TABLE_STAGES);
    for (auto& sg : p->stages) {
        const size_t bytes = set_bytes;
        e = cudaHostAlloc((void**)&sg.buf, bytes > 0 ? bytes : 1, cudaHostAllocDefault);
        if (e != cudaSuccess) return bail(fail(MLORA_ERR_OOM, "pinned table staging: %s", cudaGetErrorString(e)));
        e = cudaEventCreateWithFlags(&sg.done, cudaEventDisableTiming);
        if (e != cudaSuccess) return bail(cuda_fail(e, "cudaEventCreate"));
    }
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaDeviceSynchronize"));
    *out = p;
    return MLORA_OK;
}

mlora_status mlora_pool_destroy(mlora_pool_t p) {
    if (!p) return MLORA_OK;
    DeviceGuard g(p->device);
    if (p->last_reader) {
        if (p->reader_pending) cudaEventSynchronize(p->last_reader);
        cudaEventDestroy(p->last_reader);
    }
    if (p->copy_stream) {
        cudaStreamSynchronize(p->copy_stream);
        cudaStreamDestroy(p->copy_stream);
    }
    for (auto& kv : p->cold) {
        if (kv.second.down) cudaFreeHost(kv.second.down);
        if (kv.second.up) cudaFreeHost(kv.second.up);
        if (kv.second.busy) cudaEventDestroy(kv.second.busy);
    }
    for (auto& q : p->quarantine) cudaEventDestroy(q.free_at);
    for (auto& sg : p->stages) {
        if (sg.buf) cudaFreeHost(sg.buf);
        if (sg.done) cudaEventDestroy(sg.done);
    }
    if (p->tables_ready) cudaEventDestroy(p->tables_ready);
    for (int k = 0; k < 2; ++k)
        if (p->set_retired[k]) cudaEventDestroy(p->set_retired[k]);
    if (p->ws_base) cudaFree(p->ws_base);
    if (p->table_base) cudaFree(p->table_base);
    if (p->arena_base) cudaFree(p->arena_base);
    delete p;
    return MLORA_OK;
}

mlora_status mlora_load_adapter(mlora_pool_t p, int slot, const void* down, const void* up, int rank,
                                float scale) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    if (rank < 1 || rank > p->max_rank) return fail(MLORA_ERR_RANK, "rank %d not in [1, %d]", rank, p->max_rank);
    if (!down || !up) return fail(MLORA_ERR_INVALID_ARG, "down/up is NULL");
    SlotHost& h = p->slots[slot];
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    mlora_status st = wait_readers(p);
    if (st == MLORA_OK) st = reclaim(p, true);   // blocks of earlier prefetch evictions
    if (st != MLORA_OK) return st;
    const int need = Arena::round8(rank);
    const int have = p->arena.free_units() + (h.rank > 0 ? Arena::round8(h.rank) : 0);
    if (need > have)
        return fail(MLORA_ERR_OOM, "rank budget: adapter needs %d units, %d free (of %d)", need, have, p->units);

    if (h.rank > 0) {
        p->arena.release(slot);
        --p->loaded;
    }
    int unit = p->arena.alloc(slot, rank);
    if (unit < 0) {
        for (const ArenaMove& m : p->arena.compact()) {
            st = move_units(p, m.from, m.to, m.size);
            if (st != MLORA_OK) return st;
            p->slots[m.id].unit = m.to;
            st = push_slot(p, m.id);
            if (st != MLORA_OK) return st;
        }
        st = push_chunks(p);
        if (st != MLORA_OK) return st;
        unit = p->arena.alloc(slot, rank);
        if (unit < 0) return fail(MLORA_ERR_OOM, "arena placement failed after compaction");
    }
    const int rpad = Arena::round8(rank);
    char* dst_down = p->arena_down + (size_t)unit * p->din * p->esize;
    char* dst_up = p->arena_up + (size_t)unit * p->dout * p->esize;
    CU_TRY(cudaMemsetAsync(dst_down, 0, (size_t)rpad * p->din * p->esize, p->copy_stream));
    CU_TRY(cudaMemsetAsync(dst_up, 0, (size_t)rpad * p->dout * p->esize, p->copy_stream));
    CU_TRY(cudaMemcpyAsync(dst_down, down, (size_t)rank * p->din * p->esize, cudaMemcpyDefault, p->copy_stream));
    // Up [dout x rank] goes in blocks of 8 rank columns, each [dout x 8] row-major
    for (int g = 0; g * 8 < rank; ++g) {
        const int w = (rank - 8 * g) < 8 ? (rank - 8 * g) : 8;
        CU_TRY(cudaMemcpy2DAsync(dst_up + (size_t)g * p->dout * 8 * p->esize, 8 * p->esize,
                                 (const char*)up + (size_t)8 * g * p->esize, (size_t)rank * p->esize,
                                 (size_t)w * p->esize, (size_t)p->dout, cudaMemcpyDefault, p->copy_stream));
    }
    h.rank = rank;
    h.rpad = rpad;
    h.scale = scale;
    h.unit = unit;
    h.version += 1;
    h.chunk_rows.clear();   // an adapter of the whole layer
    ++p->loaded;
    st = push_slot(p, slot);
    if (st != MLORA_OK) return st;
    return push_chunks(p);
}

mlora_status mlora_load_adapter_modules(mlora_pool_t p, int slot, int n, const int* row_offset, const int* rows,
                                        const void* const* down, const void* const* up, const int* rank,
                                        const float* scale) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    if (n < 1 || !row_offset || !rows || !down || !up || !rank || !scale)
        return fail(MLORA_ERR_INVALID_ARG, "bad module arrays");
    // The combined adapter: module m takes rank columns [col[m], col[m] + round16(rank[m]))
    // (whole chunks, so that every chunk belongs to one module); Down stacks the
    // modules' rows, Up places module m's [rows[m] x rank[m]] at its output rows and
    // its columns, zero elsewhere.
    int R = 0;
    float common = 0.f;
    bool same = true;
    std::vector<int> col(n, 0);
    for (int m = 0; m < n; ++m) {
        if (rank[m] < 0 || rows[m] < 0 || row_offset[m] < 0 || row_offset[m] + rows[m] > p->dout)
            return fail(MLORA_ERR_INVALID_ARG, "module %d: rows [%d, %d) or rank %d out of range", m, row_offset[m],
                        row_offset[m] + rows[m], rank[m]);
        if (rank[m] == 0) continue;
        if (!down[m] || !up[m]) return fail(MLORA_ERR_INVALID_ARG, "module %d: down/up is NULL", m);
        col[m] = R;
        R += (rank[m] + CHUNK - 1) / CHUNK * CHUNK;
        if (common == 0.f) common = scale[m];
        else if (scale[m] != common) same = false;
    }
    if (R < 1 || R > p->max_rank) return fail(MLORA_ERR_RANK, "combined rank %d not in [1, %d]", R, p->max_rank);
    const size_t es = p->esize;
    std::vector<char> dc((size_t)R * p->din * es, 0), uc((size_t)p->dout * R * es, 0);
    std::vector<std::pair<int, int>> chunk_rows(R / CHUNK);
    for (int m = 0; m < n; ++m) {
        if (rank[m] == 0) continue;
        CU_TRY(cudaMemcpy(dc.data() + (size_t)col[m] * p->din * es, down[m], (size_t)rank[m] * p->din * es,
                          cudaMemcpyDefault));
        CU_TRY(cudaMemcpy2D(uc.data() + ((size_t)row_offset[m] * R + col[m]) * es, (size_t)R * es, up[m],
                            (size_t)rank[m] * es, (size_t)rank[m] * es, (size_t)rows[m], cudaMemcpyDefault));
        if (!same) {   // per-module scales differ: fold scale[m] into its Up (one rounding)
            for (int r = 0; r < rows[m]; ++r)
                for (int k = 0; k < rank[m]; ++k) {
                    char* e = uc.data() + ((size_t)(row_offset[m] + r) * R + col[m] + k) * es;
                    if (es == 4) {
                        float v;
                        std::memcpy(&v, e, 4);
                        v *= scale[m];
                        std::memcpy(e, &v, 4);
                    } else {
                        uint16_t b;
                        std::memcpy(&b, e, 2);
                        b = f32_to_bf16_rne(bf16_to_f32(b) * scale[m]);
                        std::memcpy(e, &b, 2);
                    }
                }
        }
        for (int c = col[m] / CHUNK; c < (col[m] + rank[m] + CHUNK - 1) / CHUNK; ++c)
            chunk_rows[c] = {row_offset[m], row_offset[m] + rows[m]};
    }
    mlora_status st = mlora_load_adapter(p, slot, dc.data(), uc.data(), R, same ? common : 1.f);
    if (st != MLORA_OK) return st;
    p->slots[slot].chunk_rows = chunk_rows;
    return push_chunks(p);
}

mlora_status mlora_unload_adapter(mlora_pool_t p, int slot) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    SlotHost& h = p->slots[slot];
    if (h.rank <= 0) return fail(MLORA_ERR_NOT_LOADED, "slot %d holds no adapter", slot);
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    mlora_status st = wait_readers(p);
    if (st == MLORA_OK) st = reclaim(p, true);
    if (st != MLORA_OK) return st;
    p->arena.release(slot);
    h = SlotHost{0, 0, 0.f, -1, h.version + 1};
    --p->loaded;
    st = push_slot(p, slot);
    if (st != MLORA_OK) return st;
    return push_chunks(p);
}

mlora_status mlora_host_adapter_add(mlora_pool_t p, int id, const void* down, const void* up, int rank,
                                   float scale) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (rank < 1 || rank > p->max_rank) return fail(MLORA_ERR_RANK, "rank %d not in [1, %d]", rank, p->max_rank);
    if (!down || !up) return fail(MLORA_ERR_INVALID_ARG, "down/up is NULL");
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    if (p->cold.count(id)) {   // replacing: the old copy goes first
        const mlora_status st = mlora_host_adapter_remove(p, id);
        if (st != MLORA_OK) return st;
    }
    mlora_pool::HostAdapter ha;
    ha.rank = rank;
    ha.rpad = Arena::round8(rank);
    ha.scale = scale;
    const size_t db = (size_t)ha.rpad * p->din * p->esize, ub = (size_t)ha.rpad * p->dout * p->esize;
    auto drop = [&](mlora_status s) {
        if (ha.down) cudaFreeHost(ha.down);
        if (ha.up) cudaFreeHost(ha.up);
        if (ha.busy) cudaEventDestroy(ha.busy);
        return s;
    };
    cudaError_t e = cudaHostAlloc((void**)&ha.down, db, cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaHostAlloc((void**)&ha.up, ub, cudaHostAllocDefault);
    if (e != cudaSuccess) return drop(fail(MLORA_ERR_OOM, "pinned host tier: %s", cudaGetErrorString(e)));
    std::memset(ha.down, 0, db);
    std::memset(ha.up, 0, ub);
    // Down as its rows; Up [dout x rank] in blocks of 8 rank columns, each [dout x 8]
    // (the arena's layout, so that a prefetch is two plain copies)
    e = cudaMemcpy(ha.down, down, (size_t)rank * p->din * p->esize, cudaMemcpyDefault);
    for (int b = 0; e == cudaSuccess && b * 8 < rank; ++b) {
        const int w = (rank - 8 * b) < 8 ? (rank - 8 * b) : 8;
        e = cudaMemcpy2D(ha.up + (size_t)b * p->dout * 8 * p->esize, 8 * p->esize,
                         (const char*)up + (size_t)8 * b * p->esize, (size_t)rank * p->esize, (size_t)w * p->esize,
                         (size_t)p->dout, cudaMemcpyDefault);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ha.busy, cudaEventDisableTiming);
    if (e != cudaSuccess) return drop(cuda_fail(e, "host tier copy"));
    p->cold[id] = ha;
    return MLORA_OK;
}

mlora_status mlora_host_adapter_remove(mlora_pool_t p, int id) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    auto it = p->cold.find(id);
    if (it == p->cold.end()) return fail(MLORA_ERR_NOT_LOADED, "no host-tier adapter %d", id);
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    mlora_pool::HostAdapter& ha = it->second;
    if (ha.busy_pending) CU_TRY(cudaEventSynchronize(ha.busy));   // a prefetch may still copy out of it
    cudaFreeHost(ha.down);
    cudaFreeHost(ha.up);
    cudaEventDestroy(ha.busy);
    p->cold.erase(it);
    return MLORA_OK;
}

mlora_status mlora_prefetch(mlora_pool_t p, int slot, int id, mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    auto it = p->cold.find(id);
    if (it == p->cold.end()) return fail(MLORA_ERR_NOT_LOADED, "no host-tier adapter %d", id);
    mlora_pool::HostAdapter& ha = it->second;
    SlotHost& h = p->slots[slot];
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    mlora_status rs = reclaim(p, false);
    if (rs == MLORA_OK && p->arena.free_units() < ha.rpad) rs = reclaim(p, true);
    if (rs != MLORA_OK) return rs;

    // Placement.  Normally the new copy goes to free units while the slot's current
    // block stays allocated under a quarantine id, since forwards already enqueued
    // may still read it; it returns to the allocator once they have finished.  When
    // only the slot's own units, or a compaction, make room, the readers are waited
    // for on the host first (the synchronous path of mlora_load_adapter).
    const bool had = h.rank > 0;
    int unit = -1;
    int old_block = -1;
    if (p->arena.free_units() >= ha.rpad) {
        if (had) {
            old_block = QUARANTINE_ID0 + p->next_qid++;
            p->arena.rename(slot, old_block);
        }
        unit = p->arena.alloc(slot, ha.rank);
    } else if ((had ? h.rpad : 0) + p->arena.free_units() < ha.rpad) {
        return fail(MLORA_ERR_OOM, "rank budget: adapter needs %d units, %d free (of %d)", ha.rpad,
                    p->arena.free_units() + (had ? h.rpad : 0), p->units);
    }
    if (unit < 0) {
        rs = wait_readers(p);
        if (rs == MLORA_OK) rs = reclaim(p, true);   // the compaction below moves slot blocks only
        if (rs != MLORA_OK) return rs;
        if (old_block >= 0) p->arena.release(old_block);
        else if (had) p->arena.release(slot);
        old_block = -1;
        unit = p->arena.alloc(slot, ha.rank);
        if (unit < 0) {
            for (const ArenaMove& m : p->arena.compact()) {   // slot blocks only: the quarantine is empty
                rs = move_units(p, m.from, m.to, m.size);
                if (rs != MLORA_OK) return rs;
                p->slots[m.id].unit = m.to;
            }
            unit = p->arena.alloc(slot, ha.rank);
            if (unit < 0) return fail(MLORA_ERR_OOM, "arena placement failed after compaction");
        }
    }
    if (had) --p->loaded;

    // 1. the weights, into units that no enqueued forward reads: at once, beside them
    CU_TRY(cudaMemcpyAsync(p->arena_down + (size_t)unit * p->din * p->esize, ha.down,
                           (size_t)ha.rpad * p->din * p->esize, cudaMemcpyHostToDevice, p->copy_stream));
    CU_TRY(cudaMemcpyAsync(p->arena_up + (size_t)unit * p->dout * p->esize, ha.up,
                           (size_t)ha.rpad * p->dout * p->esize, cudaMemcpyHostToDevice, p->copy_stream));
    CU_TRY(cudaEventRecord(ha.busy, p->copy_stream));
    ha.busy_pending = true;
    // 2. the tables, into the set that forwards do not read now, once the forwards that
    //    read it before the last flip have finished; then that set becomes current
    const int target = 1 - p->cur;
    if (p->captured) {
        rs = wait_readers(p);   // graph replays are invisible to the pool's events
        if (rs != MLORA_OK) return rs;
    } else if (p->set_retired_pending[target]) {
        CU_TRY(cudaStreamWaitEvent(p->copy_stream, p->set_retired[target], 0));
    }
    h.rank = ha.rank;
    h.rpad = ha.rpad;
    h.scale = ha.scale;
    h.unit = unit;
    h.version += 1;
    h.chunk_rows.clear();   // an adapter of the whole layer
    ++p->loaded;
    rs = push_tables_async(p, target);
    if (rs != MLORA_OK) return rs;
    CU_TRY(cudaEventRecord(p->tables_ready, p->copy_stream));
    // the current set's readers: everything enqueued on the caller's stream so far
    CU_TRY(cudaEventRecord(p->set_retired[p->cur], st));
    p->set_retired_pending[p->cur] = true;
    if (old_block >= 0) {   // the evicted block is named only by the retiring set
        cudaEvent_t ev;
        CU_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
        CU_TRY(cudaEventRecord(ev, st));
        p->quarantine.push_back({old_block, ev});
    }
    p->cur = target;
    p->d_slots = p->set_slots[target];
    p->d_chunks = p->set_chunks[target];
    p->ws.chunks = p->d_chunks;
    // 3. later work on the caller's stream runs with the adapter in place
    CU_TRY(cudaStreamWaitEvent(st, p->tables_ready, 0));
    return MLORA_OK;
}

mlora_status mlora_adapter_version(mlora_pool_t p, int slot, uint64_t* version) {
    if (!p || !version) return fail(MLORA_ERR_INVALID_ARG, "pool/version is NULL");
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    *version = p->slots[slot].version;
    return MLORA_OK;
}

// A quantized base weight read by the decode projection itself (codes, scales, codebook).
struct QuantW {
    int qmode;   // 1 int8 codes, per-row scale; 2 4-bit codes, per-(row, 64 columns) scale, codebook
    const void* codes;
    const float* scale;
    const float* codebook;   // host [16] (qmode 2)
};

// The forward over W (bf16 or fp32) or, with q, over a quantized W on the tensor-core
// decode path.  Arguments already checked by the callers.
static mlora_status forward_impl(mlora_pool_t p, const void* X, const void* W, const int32_t* row_adapter, int T,
                                 void* Y, mlora_stream_t stream, const QuantW* q) {
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    const bool lora = row_adapter != nullptr && p->max_slots > 0;
    const bool bf16 = p->dtype == MLORA_BF16;
    const bool tc = bf16 && tc_supported(p->dims, T);
    // the tensor-core shrink builds the segments itself; otherwise a separate segment
    // kernel runs (fp32 path, or nothing loaded: only the status bit)
    if (lora && (!tc || p->n_chunks == 0)) CU_TRY(launch_seg_build(row_adapter, T, p->d_slots, p->ws, p->dims, st));
    if (tc) {
        TcForwardArgs a{};
        a.X = X;
        a.W = W;
        a.Y = Y;
        a.T = T;
        a.lora = lora;
        a.row_adapter = row_adapter;
        a.slots = p->d_slots;
        a.maps = p->maps;
        a.arena_down = p->arena_down;
        a.ws = p->ws;
        a.dims = p->dims;
        a.n_chunks = p->n_chunks;
        a.tile_span = p->tile_span;
        a.run_stride = p->run_stride;
        a.arena_up = p->arena_up;
        a.units = p->units;
        a.n_loaded = p->loaded;
        a.stamps = p->prof_stamps;
        a.stamp_cap = p->prof_cap;
        if (q) {
            a.qmode = q->qmode;
            a.Wq = q->codes;
            a.qscale = q->scale;
            for (int i = 0; i < 16; ++i) a.qcb[i] = q->codebook ? q->codebook[i] : 0.f;
        }
        CU_TRY(tc_forward(a, st));
    } else {
        if (lora) CU_TRY(launch_shrink_simt(bf16, X, row_adapter, T, p->d_slots, p->arena_down, p->ws, p->dims, st));
        CU_TRY(launch_base_expand_simt(bf16, X, W, row_adapter, T, Y, p->d_slots, p->arena_up, p->ws, p->dims, lora, st));
    }
    if (lora) p->last_T = T;
    return note_reader(p, st);
}

mlora_status mlora_forward(mlora_pool_t p, const void* X, const void* W, const int32_t* row_adapter, int T,
                           void* Y, mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (T < 0 || T > p->max_tokens) return fail(MLORA_ERR_INVALID_ARG, "T %d not in [0, %d]", T, p->max_tokens);
    if (T == 0) return MLORA_OK;
    if (!X || !W || !Y) return fail(MLORA_ERR_INVALID_ARG, "X/W/Y is NULL");
    if (p->dtype == MLORA_BF16 && (!aligned16(X) || !aligned16(W) || !aligned16(Y)))
        return fail(MLORA_ERR_INVALID_ARG, "bf16 X/W/Y must be 16-byte aligned");
    return forward_impl(p, X, W, row_adapter, T, Y, stream, nullptr);
}

// W <- W + sign * scale * Up Down of the adapter in `slot` (merge: +1, un-merge: -1).
static mlora_status merge_signed(mlora_pool_t p, void* W, int slot, float sign, mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (!W) return fail(MLORA_ERR_INVALID_ARG, "W is NULL");
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    if (p->slots[slot].rank <= 0) return fail(MLORA_ERR_NOT_LOADED, "slot %d holds no adapter", slot);
    if (p->dtype == MLORA_BF16 && !aligned16(W)) return fail(MLORA_ERR_INVALID_ARG, "bf16 W must be 16-byte aligned");
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    if (p->dtype == MLORA_BF16)   // tensor cores (MMA over the rank, W tile in and out by TMA)
        CU_TRY(launch_merge_tc(W, p->d_slots, slot, p->maps, p->ws.status, p->dims, sign, st));
    else
        CU_TRY(launch_merge_simt(false, W, p->d_slots, slot, p->arena_down, p->arena_up, p->dims, sign, st));
    return note_reader(p, st);
}

mlora_status mlora_merge(mlora_pool_t p, void* W, int slot, mlora_stream_t stream) {
    return merge_signed(p, W, slot, 1.f, stream);
}

mlora_status mlora_unmerge(mlora_pool_t p, void* W, int slot, mlora_stream_t stream) {
    return merge_signed(p, W, slot, -1.f, stream);
}

mlora_status mlora_dequantize(const void* Wq, const float* row_scale, int dout, int din, mlora_dtype dtype, void* W,
                              mlora_stream_t stream) {
    if (!Wq || !row_scale || !W) return fail(MLORA_ERR_INVALID_ARG, "Wq/row_scale/W is NULL");
    if (dout < 0 || din < 0) return fail(MLORA_ERR_INVALID_ARG, "negative size");
    if (dtype != MLORA_BF16 && dtype != MLORA_F32) return fail(MLORA_ERR_INVALID_ARG, "bad dtype");
    if (!aligned16(Wq) || !aligned16(W)) return fail(MLORA_ERR_INVALID_ARG, "Wq and W must be 16-byte aligned");
    CU_TRY(launch_dequant(dtype == MLORA_BF16, (const int8_t*)Wq, row_scale, dout, din, W, (cudaStream_t)stream));
    return MLORA_OK;
}

mlora_status mlora_forward_quantized(mlora_pool_t p, const void* X, const void* Wq, const float* row_scale,
                                     void* W_scratch, const int32_t* row_adapter, int T, void* Y,
                                     mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (T < 0 || T > p->max_tokens) return fail(MLORA_ERR_INVALID_ARG, "T %d not in [0, %d]", T, p->max_tokens);
    if (T == 0) return MLORA_OK;
    if (p->dtype == MLORA_BF16 && tc_quantized_fits(p->dims, T, false)) {
        // decode-sized batch: the projection reads the codes and restores each W tile in
        // shared memory (no restore pass over W; W_scratch is not used)
        if (!X || !Wq || !row_scale || !Y) return fail(MLORA_ERR_INVALID_ARG, "X/Wq/row_scale/Y is NULL");
        if (!aligned16(X) || !aligned16(Wq) || !aligned16(Y))
            return fail(MLORA_ERR_INVALID_ARG, "X/Wq/Y must be 16-byte aligned");
        const QuantW q{1, Wq, row_scale, nullptr};
        return forward_impl(p, X, nullptr, row_adapter, T, Y, stream, &q);
    }
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    mlora_status st = mlora_dequantize(Wq, row_scale, p->dout, p->din, p->dtype, W_scratch, stream);
    if (st != MLORA_OK) return st;
    return mlora_forward(p, X, W_scratch, row_adapter, T, Y, stream);
}

mlora_status mlora_merge_quantized(mlora_pool_t p, void* Wq, float* row_scale, int slot, mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (!Wq || !row_scale) return fail(MLORA_ERR_INVALID_ARG, "Wq/row_scale is NULL");
    if (!aligned16(Wq)) return fail(MLORA_ERR_INVALID_ARG, "Wq must be 16-byte aligned");
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    if (p->slots[slot].rank <= 0) return fail(MLORA_ERR_NOT_LOADED, "slot %d holds no adapter", slot);
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    // bf16 pools with whole 16-byte code rows: tensor cores (merged rows' max, new codes,
    // new scales); otherwise CUDA cores, the merged rows held in shared memory
    const bool tensor_cores = p->dtype == MLORA_BF16 && p->din % 16 == 0;
    const cudaError_t e = tensor_cores
                              ? launch_merge_quant_tc((int8_t*)Wq, row_scale, p->row_max, p->d_slots, slot, p->maps,
                                                      p->ws.status, p->dims, st)
                              : launch_merge_quant(p->dtype == MLORA_BF16, (int8_t*)Wq, row_scale, p->d_slots, slot,
                                                   p->arena_down, p->arena_up, p->dims, st);
    if (e == cudaErrorInvalidValue && !tensor_cores)
        return fail(MLORA_ERR_INVALID_ARG, "din %d too large for the quantized merge", p->din);
    if (e != cudaSuccess) return cuda_fail(e, tensor_cores ? "quantized merge (tensor cores)" : "quantized merge");
    return note_reader(p, st);
}

mlora_status mlora_dequantize_nf4(const void* codes, const float* absmax, const float* codebook, int dout, int din,
                                  mlora_dtype dtype, void* W, mlora_stream_t stream) {
    if (!codes || !absmax || !codebook || !W) return fail(MLORA_ERR_INVALID_ARG, "codes/absmax/codebook/W is NULL");
    if (dout < 0 || din < 0 || din % 64 != 0) return fail(MLORA_ERR_INVALID_ARG, "din %d must be a multiple of 64", din);
    if (dtype != MLORA_BF16 && dtype != MLORA_F32) return fail(MLORA_ERR_INVALID_ARG, "bad dtype");
    if (!aligned16(codes) || !aligned16(W)) return fail(MLORA_ERR_INVALID_ARG, "codes and W must be 16-byte aligned");
    CU_TRY(launch_dequant_nf4(dtype == MLORA_BF16, (const uint8_t*)codes, absmax, codebook, dout, din, W,
                              (cudaStream_t)stream));
    return MLORA_OK;
}

mlora_status mlora_forward_nf4(mlora_pool_t p, const void* X, const void* codes, const float* absmax,
                               const float* codebook, void* W_scratch, const int32_t* row_adapter, int T, void* Y,
                               mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (T < 0 || T > p->max_tokens) return fail(MLORA_ERR_INVALID_ARG, "T %d not in [0, %d]", T, p->max_tokens);
    if (T == 0) return MLORA_OK;
    if (!X || !codes || !absmax || !codebook || !Y) return fail(MLORA_ERR_INVALID_ARG, "X/codes/absmax/codebook/Y is NULL");
    if (p->din % 64 != 0) return fail(MLORA_ERR_INVALID_ARG, "din %d must be a multiple of 64", p->din);
    if (!aligned16(X) || !aligned16(codes) || !aligned16(Y))
        return fail(MLORA_ERR_INVALID_ARG, "X/codes/Y must be 16-byte aligned");
    if (p->dtype == MLORA_BF16 && tc_quantized_fits(p->dims, T, true) && aligned16(absmax)) {
        const QuantW q{2, codes, absmax, codebook};
        return forward_impl(p, X, nullptr, row_adapter, T, Y, stream, &q);
    }
    if (!W_scratch)
        return fail(MLORA_ERR_INVALID_ARG, "W_scratch is NULL (needed unless bf16, T <= 256, dout %% 4 == 0 and absmax "
                                           "16-byte aligned)");
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    mlora_status st = mlora_dequantize_nf4(codes, absmax, codebook, p->dout, p->din, p->dtype, W_scratch, stream);
    if (st != MLORA_OK) return st;
    return mlora_forward(p, X, W_scratch, row_adapter, T, Y, stream);
}

mlora_status mlora_merge_nf4(mlora_pool_t p, void* codes, float* absmax, const float* codebook, int slot,
                             mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (!codes || !absmax || !codebook) return fail(MLORA_ERR_INVALID_ARG, "codes/absmax/codebook is NULL");
    if (p->din % 64 != 0) return fail(MLORA_ERR_INVALID_ARG, "din %d must be a multiple of 64", p->din);
    if (slot < 0 || slot >= p->max_slots) return fail(MLORA_ERR_BAD_SLOT, "slot %d not in [0, %d)", slot, p->max_slots);
    if (p->slots[slot].rank <= 0) return fail(MLORA_ERR_NOT_LOADED, "slot %d holds no adapter", slot);
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    CU_TRY(launch_merge_nf4(p->dtype == MLORA_BF16, (uint8_t*)codes, absmax, codebook, p->d_slots, slot,
                            p->arena_down, p->arena_up, p->dims, st));
    return note_reader(p, st);
}

mlora_status mlora_pool_status(mlora_pool_t p, mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    CU_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    uint32_t word = 0;
    CU_TRY(cudaMemcpyAsync(&word, p->ws.status, sizeof word, cudaMemcpyDeviceToHost, p->copy_stream));
    CU_TRY(cudaMemsetAsync(p->ws.status, 0, sizeof word, p->copy_stream));
    CU_TRY(cudaStreamSynchronize(p->copy_stream));
    if (word & STATUS_TIMEOUT) return fail(MLORA_ERR_DEVICE_TIMEOUT, "a kernel pipeline wait gave up");
    if (word & STATUS_BAD_ROW) return fail(MLORA_ERR_DEVICE_ROW, "a row named an invalid or empty slot");
    return MLORA_OK;
}

mlora_status mlora_pool_info(mlora_pool_t p, mlora_pool_info_t* info) {
    if (!p || !info) return fail(MLORA_ERR_INVALID_ARG, "pool/info is NULL");
    info->din = p->din;
    info->dout = p->dout;
    info->dtype = (int32_t)p->dtype;
    info->max_slots = p->max_slots;
    info->max_rank = p->max_rank;
    info->max_tokens = p->max_tokens;
    info->rank_units = p->units;
    info->rank_units_used = p->arena.used();
    info->loaded = p->loaded;
    info->device = p->device;
    info->arena_bytes = p->arena_bytes;
    info->table_bytes = p->table_bytes;
    info->workspace_bytes = p->ws_bytes;
    info->ext_run_stride = p->run_stride;
    info->reserved = 0;
    return MLORA_OK;
}

mlora_status mlora_debug_segments(mlora_pool_t p, const int32_t* row_adapter, int T, int32_t* perm,
                                  int32_t* offsets, mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (T < 0 || T > p->max_tokens) return fail(MLORA_ERR_INVALID_ARG, "T %d not in [0, %d]", T, p->max_tokens);
    if (!offsets || (T > 0 && !perm)) return fail(MLORA_ERR_INVALID_ARG, "perm/offsets is NULL");
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    if (!row_adapter || p->max_slots == 0 || T == 0) {
        if (T > 0) CU_TRY(cudaMemsetAsync(perm, 0xFF, sizeof(int32_t) * (size_t)T, st));
        CU_TRY(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)(p->max_slots + 1), st));
        return MLORA_OK;
    }
    CU_TRY(launch_seg_build(row_adapter, T, p->d_slots, p->ws, p->dims, st));
    p->last_T = -1;   // the workspace now holds this builder's segments, not a forward's
    CU_TRY(cudaMemcpyAsync(perm, p->ws.perm, sizeof(int32_t) * (size_t)T, cudaMemcpyDeviceToDevice, st));
    CU_TRY(cudaMemcpyAsync(offsets, p->ws.offsets, sizeof(int32_t) * (size_t)(p->max_slots + 1),
                           cudaMemcpyDeviceToDevice, st));
    return note_reader(p, st);
}

mlora_status mlora_debug_last_segments(mlora_pool_t p, int T, int32_t* perm, int32_t* offsets,
                                       mlora_stream_t stream) {
    if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
    if (T < 0 || T > p->max_tokens) return fail(MLORA_ERR_INVALID_ARG, "T %d not in [0, %d]", T, p->max_tokens);
    if (!offsets || (T > 0 && !perm)) return fail(MLORA_ERR_INVALID_ARG, "perm/offsets is NULL");
    if (p->last_T != T) return fail(MLORA_ERR_INVALID_ARG, "the last forward with a row map had %d rows, not %d", p->last_T, T);
    DeviceGuard g(p->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    if (T > 0) CU_TRY(cudaMemcpyAsync(perm, p->ws.perm, sizeof(int32_t) * (size_t)T, cudaMemcpyDeviceToDevice, st));
    CU_TRY(cudaMemcpyAsync(offsets, p->ws.offsets, sizeof(int32_t) * (size_t)(p->max_slots + 1),
                           cudaMemcpyDeviceToDevice, st));
    return MLORA_OK;
}

mlora_status mlora_profile_stamps(mlora_pool_t p, void* records, int cap) {
    if (!p || cap < 0 || (cap > 0 && !records)) return fail(MLORA_ERR_INVALID_ARG, "bad profiling record buffer");
    if (((uintptr_t)records & 7u) != 0) return fail(MLORA_ERR_INVALID_ARG, "record buffer must be 8-byte aligned");
    p->prof_stamps = cap > 0 ? (unsigned long long*)records : nullptr;
    p->prof_cap = cap;
    return MLORA_OK;
}

}  // extern "C"
