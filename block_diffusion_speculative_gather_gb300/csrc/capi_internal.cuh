// Host accessors of a context for the C-ABI source files other than the one
// that defines the context (the many-sequence round builds on contexts).
#pragma once

#include <cudaTypedefs.h>

#include "../../include/dflash.h"
#include "common.cuh"

namespace dfl {

DevState* ctx_state(const dflash_ctx* c);               // device round state
// device RoPE angles of every cache position: cos, sin [rows][head_dim/2]
void rope_table(const dflash_ctx* c, const float** cos_tab, const float** sin_tab, int* rows);
const dflash_layer* ctx_layers(const dflash_ctx* c, bool target);   // host copies
// the context's copy of every draft layer's [W_k; W_v] (bf16, rows in layer
// order) and k-norm weights [layers][head_dim]; false when it has none
bool ctx_grouped_ctxkv(const dflash_ctx* c, const void** w, const float** k_norm, int* rows);
const dflash_weights& ctx_weights(const dflash_ctx* c);
// 2D tensor map over a row-major [rows][inner] matrix of es-byte elements.
int encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int es, uint64_t inner,
               uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz);

}  // namespace dfl
