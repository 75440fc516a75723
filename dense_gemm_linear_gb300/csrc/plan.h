// Host-side planner interface (pure host code).
#pragma once

#include <cstdint>

#include "dgl.h"

namespace dgl {

constexpr int64_t kDecodeMaxM = 16;

void tile_metrics(int64_t m, int64_t n, int tile_m, int tile_n, int units, dgl_plan_info* out);
double operand_bytes(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K);
int tc_tile_k(int dtype);
int tc_stages(int tile_n);
bool tc_supported_tile(int tile_m, int tile_n);
void fill_tc_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int tile_m, int tile_n, int num_sms,
                  dgl_plan_info* out);
void fill_decode_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out);
int decode_grid(int64_t n, int num_sms);
void choose_plan(int dtype, int out_dtype, int64_t m, int64_t n, int64_t K, int num_sms, dgl_plan_info* out);

}  // namespace dgl
