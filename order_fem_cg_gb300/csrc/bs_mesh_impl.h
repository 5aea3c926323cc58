// bs_mesh_impl.h -- host representation of a mesh and its index tables.
#pragma once

#include <cstdint>
#include <vector>

#include "bs.h"

// Two-pass gather/scatter plan: the permutation between global (CSR) order
// and local order done through shared memory in two coalesced passes.
//
// Scatter (q_L = Z q_G): pass 1 takes a tile of consecutive global rows,
// holds their q_G values in shared memory and writes, for every bucket of
// consecutive locals, one contiguous run of the work array; pass 2 takes one
// bucket's runs, places them by local offset in shared memory and writes the
// bucket's q_L range coalesced.  Gather (q_G = Z^T q_L) mirrors it: pass 1
// tiles consecutive locals, buckets are ranges of consecutive rows; pass 2
// places a bucket's values by CSR position and sums each row in ascending
// local order.  The work array is ordered bucket-major, then tile, so both
// passes touch it in runs.
//
// Each tile and bucket is handled by a cluster of `cluster` thread blocks
// whose shared memories together hold it (distributed shared memory), so
// a tile is cluster x the per-block size; runs grow with tile x bucket.
// A gather bucket is `cluster` consecutive sub-buckets, each a row range
// of at most g_bucket_entries entries and rows held by one block.  Inside a
// sub-bucket the values are staged grouped by row length m: the R rows
// with m entries form an m x R column-major block (entry j of the group's
// q-th row at j R + q, rows in ascending order), so that a warp sums rows
// of equal length with all lanes busy -- a binary64 warp instruction holds
// the SM's FP64 pipe for ~20 cycles on GB300 however many lanes are
// active -- and its lanes read consecutive shared-memory words.
// Sizes below are per block.
struct bs_plan {
    bool valid = false;
    int32_t cluster = 1;
    int32_t s_tile_rows = 0, s_bucket_len = 0, g_tile_len = 0, g_bucket_entries = 0;
    int32_t s_ntiles = 0, s_nbuckets = 0, g_ntiles = 0, g_nbuckets = 0;
    int32_t g_bucket_rows_max = 0, g_bucket_entries_max = 0;  // per sub-bucket
    int32_t g_mmax = 0;                                       // longest row
    std::vector<int32_t> s_tileRows;   // [s_ntiles+1]  first row of each scatter tile
    std::vector<int32_t> s_runStart;   // [(s_ntiles+1) x s_nbuckets] work position of run (t, b)
    std::vector<uint16_t> s_src;       // [nnz] tile-major: row offset within the tile,
                                       // | BS_PLAN_RUN_START on a run's first slot
    std::vector<uint16_t> s_dst;       // [nnz] work order: local offset within the bucket
    std::vector<int32_t> g_subRows;    // [cluster x g_nbuckets + 1] first row of each sub-bucket
    std::vector<int32_t> g_tileSlot;   // [g_ntiles+1]  unmasked locals before each tile
    std::vector<int32_t> g_runStart;   // [(g_ntiles+1) x g_nbuckets]
    std::vector<uint16_t> g_src;       // [nnz] tile-major: local offset within the tile,
                                       // | BS_PLAN_RUN_START on a run's first slot
    std::vector<uint16_t> g_pos;       // [nnz] work order: staged position within the bucket
    std::vector<uint16_t> g_groupStart; // [cluster x g_nbuckets x (g_mmax+1)] per sub-bucket:
                                        // [m-1] = first position of the rows of length m,
                                        // [g_mmax] = entries of the sub-bucket
    std::vector<uint16_t> g_rowPos;    // [NG] staged position of a row's first value within
                                       // its sub-bucket (where its sum is left), 0xFFFF for a
                                       // row without entries
};

struct bs_mesh {
    int32_t E = 0, N = 0;
    uint32_t flags = 0;
    int32_t max_row = 0, seg_max = 0, seg_target = 0;
    int64_t K = 0, NL = 0, NG = 0, nnz = 0;
    std::vector<int32_t> scatterIds, rowStarts, localIds, blockStarts;
    bs_plan plan;
};

// Default plan: one block per tile or bucket (clusters of 2 and 4 measured
// slower on GB300: random 8-byte accesses to a peer block's shared memory
// cost more than the longer runs save), each block filling most of a GB300
// SM's 227 KB of shared memory (8 bytes per staged value).
constexpr int32_t BS_TILE_CLUSTER = 1;
constexpr int32_t BS_TILE_S_ROWS = 24576;
constexpr int32_t BS_TILE_S_BUCKET = 24576;
constexpr int32_t BS_TILE_G_LOCALS = 24576;
constexpr int32_t BS_TILE_G_BUCKET = 22528;
// Largest dynamic shared memory of one block.
constexpr int64_t BS_SMEM_MAX = 232448;

// Shared-memory bytes the four plan kernels need.
int64_t bs_plan_smem_s1(const bs_plan &p);
int64_t bs_plan_smem_s2(const bs_plan &p);
int64_t bs_plan_smem_g1(const bs_plan &p);
int64_t bs_plan_smem_g2(const bs_plan &p);
// Host-side fault injection, for tests of a caller's error handling: the
// comma-separated names in the environment variable BS_FAULT select the
// failures to fake -- "alloc": bs_ctx_create reports BS_ENOMEM before
// touching the device; "launch": every launching call reports BS_ECUDA
// without launching; "badtable": the mesh builders corrupt one scatterIds
// and one localIds entry (out of range) after building.  Nothing of this
// faults a GPU; the device kernels' own bounds checks turn a bad table into
// BS_EBOUNDS.  Reads the environment at every call.
bool bs_fault(const char *what);

// Marks the first slot of a run in s_src / g_src (tile offsets are < 2^15).
constexpr uint32_t BS_PLAN_RUN_START = 0x8000u;

// Longest row the grouped gather supports.
constexpr int32_t BS_PLAN_MMAX = 32;

// (Re)builds m->plan; leaves it invalid (empty) when a kernel would need
// more shared memory than a block can have.  Throws std::bad_alloc.
void bs_plan_build(bs_mesh *m, int32_t s_tile_rows, int32_t s_bucket_len, int32_t g_tile_len,
                   int32_t g_bucket_entries, int32_t cluster);
