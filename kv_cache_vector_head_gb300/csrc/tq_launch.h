// Host-side launchers of libtq's kernels (defined in the .cu files).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tq_device.cuh"

namespace tq {

cudaError_t launch_quantize_flat(const KParams& P, const void* x, int dtype, long long n_vec, bool is_key,
                                 uint32_t* codes, uint32_t* signs, float* norms, float* rnorms, cudaStream_t st);
cudaError_t launch_append_direct(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                 long long n_tok, const long long* slots, cudaStream_t st);
// Whole sequences of seq_tok tokens: n_c into their pages, the rest into the window ring, counters set.
cudaError_t launch_prefill_cache(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                 int seq_tok, int n_c, cudaStream_t st);
cudaError_t launch_append_step(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                               cudaStream_t st);

// Decode workspace layout (byte offsets; every region 256-byte aligned).
struct WsLayout {
  size_t afrag, ml, acc, total;
  size_t afrag_bytes_per_head;  // per (sequence, kv head)
  int n_comp_splits;   // compressed-page splits; one extra split holds the window
  int pages_per_split;
};
WsLayout decode_ws_layout(const KParams& P, int batch, int max_ctx, int n_splits, int num_sms);

cudaError_t launch_decode(const KParams& P, const KCache& C, const void* q, int dtype, float scale, float* out,
                          float* lse, float* scores, void* ws, const WsLayout& L, int max_ctx, cudaStream_t st);

// Virtual sequences of a prefill chunk: query i of sequence b is row v = b n_query + i,
// visible length seq_len[b] - n_query + i + 1, its compressed part clipped to it.
cudaError_t launch_prefill_virtual(const KCache& C, int n_query, int32_t* seq_v, int32_t* nc_v, int32_t* parent,
                                   cudaStream_t st);

// Prefill attention with query tiles: 16 (query, head) rows of a chunk per CTA share every page
// (TurboQuant_prod keys with 2 or 4 Walsh planes, values of 2..4 bits, no mixed-channel keys or
// byte norms, d = 128 or 256).  V is the chunk's virtual-sequence cache; the workspace layout
// takes prefill_tile_splits() compressed splits.
bool prefill_tiles_ok(const KParams& P);
int prefill_tile_splits(const KParams& P, int batch, int n_query, int max_ctx, int num_sms);
cudaError_t launch_prefill_tiles(const KParams& P, const KCache& V, int n_query, int batch, const void* q, int dtype,
                                 float scale, float* out, float* lse, void* ws, const WsLayout& L, int max_ctx,
                                 cudaStream_t st);

cudaError_t read_clear_quant_error(unsigned* bits);
cudaError_t read_clear_decode_error(unsigned* bits);
#ifdef TQ_TEST_HOOKS
cudaError_t set_test_wait_fault(int on);
#endif

}  // namespace tq
