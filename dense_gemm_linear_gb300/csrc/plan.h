// Host-side planner interface (pure host code).
#pragma once

#include <cstdint>

#include "dgl.h"

namespace dgl {

constexpr int64_t kDecodeMaxM = 16;

void tile_metrics(int64_t m, int64_t n, int tile_m, int tile_n, int units, dgl_plan_info* out);
double operand_bytes(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K);
int tc_tile_k(int dtype);
int tc_stages(int tile_m, int tile_n);
bool tc_supported_tile(int tile_m, int tile_n);
// stream_k: -2 the planner's default (split-K tail where it applies), -1 the
// cost model decides on stream-K, 0 off, 1 stream-K over all workers (when
// eligible), S >= 2 a split-K tail over S workers per tile (when it fits).
void fill_tc_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int tile_m, int tile_n, int num_sms,
                  dgl_plan_info* out, int stream_k);
bool split_tail_eligible(int64_t m, int64_t n, int64_t K, int dtype, int tile_m, int tile_n, int num_sms);
bool stream_k_eligible(int64_t m, int64_t n, int64_t K, int dtype, int tile_m, int tile_n, int num_sms);
int tail_split_ways(int64_t m, int64_t n, int64_t K, int dtype, int tile_m, int tile_n, int num_sms);
void fill_decode_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out);
int decode_parts(int64_t n, int num_sms);
int decode_grid(int64_t n, int num_sms);
int decode_group(int rows_hi, int nk);                         // K steps stacked into one 128-row MMA operand
int decode_plane_bytes(int rows_hi, int group);               // one B slot: 128 / group rows (group 1: rows_hi
                                                              // rounded up to 8), x 128 bytes
int decode_stage_bytes(int rows_hi, int ksteps, int group);   // ksteps x (16-row A box + B slot)
int decode_stages(int rows_hi, int ksteps, int group);        // ring depth in 192 KB, at most 32
int decode_ksteps(int rows_hi, int nk, int group);            // 128-byte K steps per stage, a multiple of group
// Tiles with a linear-layer epilogue variant: 128 or 256 wide, and CTA pairs
// (tile_m 256) when gated.
bool tc_supported_epi_tile(int tile_m, int tile_n, bool gated);
// The plan of a linear layer (dgl_linear): as choose_plan, restricted to the
// tiles above; a gated layer is planned as a product with 2 n rows of B.
void choose_linear_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, bool gated, int num_sms,
                        dgl_plan_info* out);
void choose_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out);
// The block-scaled FP4 plan: 128 x 256 tiles on one CTA each.
void fill_mx_plan(int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out);

}  // namespace dgl
