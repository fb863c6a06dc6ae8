// Internal declarations shared by the libkvc translation units.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/kvc.h"

// Device-detected error bits (pool error word).
#define KVC_EBIT_BAD_BLOCK 1u
#define KVC_EBIT_RANGE 2u
#define KVC_EBIT_TIMEOUT 4u

struct kvc_pool {
    int64_t N;            // physical blocks
    int32_t bs, L, H_KV, D, dtype, s, device;   // s: bytes per element (0 for int4)
    int32_t bits;         // bits per stored element: 16, 8 or 4
    uint8_t *base;        // pool bytes
    size_t layer_bytes, pool_bytes;
    float *scales;        // [L][2][H_KV][D] (e4m3 pools)
    float *absmax;        // [L][2][H_KV][D] running absmax for kvc_calibrate_fp8
    uint32_t *err;        // device error word
    CUtensorMap tmap;     // rows of D elements; box {128 B, 2*bs rows}; 128-byte swizzle
    bool tmap_ok;
    CUtensorMap tmap16;   // same rows, box {128 B, 16 rows}: the keys or the values of 16 positions
    bool tmap16_ok;
    void *ws;             // workspace: arrival counters [ws_counters], then split / record partials
    size_t ws_bytes;      // partial bytes after the counter region
    size_t ws_counters;   // arrival counters at the front (zero between launches)
    int num_sms;
};

namespace kvc {

extern std::atomic<uint64_t> g_launches;

// Decode / prefill attention launch parameters (one layer).
struct DecodeParams {
    const uint16_t *q;       // bf16 [B][H_Q][D]
    const int32_t *bt;       // block table rows
    const int32_t *lens;     // [B] positions attended, or nullptr: len(b) = len_base + b + 1
    int64_t bt_stride;       // elements between table rows (0: every row is the same row)
    int32_t max_blocks;
    int32_t len_base;
    int32_t B, H_Q, H_KV, g;  // B = units (grid z)
    int32_t ppu;             // query positions per unit: 1 for decode, a tile of a prefill chunk
    int32_t n_pos;           // query positions in all (decode: B; prefill: n_q)
    int32_t layer;
    int32_t chunk;           // logical blocks per split (the split kernel: a multiple of 4; tcgen05: any)
    int32_t max_splits;
    int64_t N;
    float scale_log2;        // softmax scale * log2(e)
    const float *s_k;        // this layer's e4m3 scales [H_KV][D] (keys), else nullptr
    const float *s_v;        // (values)
    float *out;              // fp32 [B][H_Q][D]
    float *lse;              // fp32 [B][H_Q] or nullptr
    float *part_o;           // [B][H_Q][max_splits][D]
    float2 *part_ml;         // [B][H_Q][max_splits]  (running max in log2 units, sum)
    uint32_t *err;
    // fused append (kvc_decode_step): the step's new key / value rows, bf16 [B][H_KV][D],
    // written at position lens[b] before attending to lens[b] + 1 positions; nullptr = none
    const uint16_t *k_new;
    const uint16_t *v_new;
    uint8_t *pool;           // pool base (the fused append's global store, the L2 prefetch)
    // split-K arrival counters [B][H_KV], zero between launches; nullptr = merge in a separate kernel
    uint32_t *counters;
    // test hook (KVC_TEST_STALL set): the copy producers issue no load and never arrive, so every
    // bounded wait expires and the launch reports KVC_ERR_TIMEOUT
    int32_t stall_loads;
};

kvc_status cuda_status(cudaError_t e);
kvc_status check_device(const kvc_pool *pool);

// Launchers implemented per element type.
kvc_status launch_decode_bf16(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream);
kvc_status launch_decode_fp8(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream);
kvc_status launch_decode_int4(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream);

// Split-K sizing: blocks per split and the split count for a batch.
void choose_split(const kvc_pool *pool, int units, int max_blocks, int ctas_per_sm, int *chunk, int *max_splits,
                  int n_tiles);
// Split sizing of the tensor-memory decode kernel (whole 128-token tiles).
void choose_split_tc(const kvc_pool *pool, int units, int max_blocks, int ctas_per_sm, int unit, int *chunk,
                     int *max_splits);

// Look up (and so reserve) the allocation-free decode's scratch array for the current
// context of `device`; kvc_pool_create calls it.
void noalloc_prepare(int device);

// 8-wide query n-tiles a group of g query heads occupies in the decode kernel.
inline int n_tiles(int g) { return g <= 8 ? 1 : (g <= 16 ? 2 : 4); }

}  // namespace kvc
