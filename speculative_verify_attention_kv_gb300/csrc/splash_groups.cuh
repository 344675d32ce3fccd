// Work items and workspace layout of a plan with prefix groups (cross-sequence
// query stacking over shared prefix pages). Only the shared-prefix entry point
// plans this way; the other entry points use WorkspaceLayout.
#pragma once

#include "splash_common.cuh"

namespace splash {

// Prefix groups are planned for batches of up to this many sequences (the
// group planner keeps its per-sequence arrays in shared memory).
constexpr int kPrefixGroupMaxSeqs = 1024;

// A work item: a set of query rows of one KV head (the item's units are
// (item, KV head)) against a key range of one page-table row. Item b <
// num_seqs is sequence b (its rows t * G + g; its keys, or with a shared
// prefix only the keys after it). Items past num_seqs are row blocks of a
// prefix group: up to kMaxRows consecutive rows of the group's stacked rows
// against the group's common prefix keys.
// Row r of an item is query token qbase + (r0 + r) / G, query head
// h * G + (r0 + r) % G; it sees keys klo <= j < Lk with j <= ctx + (r0 + r) / G.
struct ItemDesc {
  int b;          // sequence whose page-table row holds the item's pages
  int qbase;      // first query token of the item's rows
  int r0;         // row offset of the item's row 0 from qbase's row 0
  int R;          // rows
  int ctx;        // causal bound of the rows (see above)
  int Lk;         // one past the last key
  int klo;        // first key, a tile boundary
  int grouped;    // 1: part of a prefix group, so its rows always go to partials
};
static_assert(sizeof(ItemDesc) == 32, "item size");

// Items of a batch of B sequences: the sequences and at most B row blocks (a
// group of m sequences is stacked only when it needs fewer than m blocks).
__host__ __device__ inline int max_items(int B) { return 2 * B; }

// Byte offsets of the workspace regions of a plan with prefix groups (all
// 256-aligned; the plan header first, as in WorkspaceLayout). Every sequence
// is in the tensor-core class.
struct GroupLayout {
  size_t q_off;        // int32 [B+1]    first token row of each sequence
  size_t seq_T;        // int32 [B]      validated block length (0 if skipped)
  size_t seq_ctx;      // int32 [B]
  size_t seq_grp;      // int2  [B]      first row-block item of the sequence's group
                       //                (-1: none), offset of its row 0 in the stacked rows
  size_t items;        // ItemDesc [2B]
  size_t stp;          // int32 [2B+1]   exclusive prefix of tiles per item; INT_MAX past the items
  size_t nseg;         // int32 [2B*Hkv] CTAs (segments) that cover the unit
  size_t cfirst;       // int32 [2B*Hkv] first CTA of the unit
  size_t part_base;    // int32 [2B*Hkv] first partial row of the unit, -1: rows go to the output
  size_t wcost;        // int64 [2B+1]   exclusive prefix of item costs
  size_t cta_start;    // int32 [kMaxCtas+1] first tile of each CTA
  size_t o_part;       // fp32  [rows_bound, D]
  size_t lse_part;     // fp32  [rows_bound]
  size_t total;
};

__host__ __device__ inline GroupLayout make_group_layout(int B, int Hkv, int D,
                                                         long long rows_bound) {
  GroupLayout L;
  const size_t NI = (size_t)max_items(B);
  size_t o = align256(sizeof(PlanHeader));
  L.q_off = o;      o = align256(o + sizeof(int) * (size_t)(B + 1));
  L.seq_T = o;      o = align256(o + sizeof(int) * (size_t)B);
  L.seq_ctx = o;    o = align256(o + sizeof(int) * (size_t)B);
  L.seq_grp = o;    o = align256(o + sizeof(int2) * (size_t)B);
  L.items = o;      o = align256(o + sizeof(ItemDesc) * NI);
  L.stp = o;        o = align256(o + sizeof(int) * (NI + 1));
  L.nseg = o;       o = align256(o + sizeof(int) * NI * Hkv);
  L.cfirst = o;     o = align256(o + sizeof(int) * NI * Hkv);
  L.part_base = o;  o = align256(o + sizeof(int) * NI * Hkv);
  L.wcost = o;      o = align256(o + sizeof(long long) * (NI + 1));
  L.cta_start = o;  o = align256(o + sizeof(int) * (size_t)(kMaxCtas + 1));
  L.o_part = o;     o = align256(o + sizeof(float) * (size_t)rows_bound * D);
  L.lse_part = o;   o = align256(o + sizeof(float) * (size_t)rows_bound);
  L.total = o;
  return L;
}

// Partial rows of a plan with prefix groups: split units hold at most
// 2 * (CTAs) segments (a CTA's range shares at most its first and its last
// unit with other CTAs) of at most max(rows_cap, kMaxRows) rows; a grouped
// unit writes partials even when one CTA covers it, and every grouped output
// row has one such row in its block and one in its own unit.
inline long long group_rows_bound(int num_q_tokens, int num_q_heads, int rows_cap, int ncta) {
  const int rows = rows_cap > kMaxRows ? rows_cap : kMaxRows;
  return 2LL * rows * ncta + 2LL * num_q_tokens * num_q_heads + 1;
}

}  // namespace splash
