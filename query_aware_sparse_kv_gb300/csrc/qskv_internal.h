// Host-side declarations shared by the C-ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qskv {

constexpr int kDtypeF32 = 0;  // matches QSKV_F32
constexpr int kDtypeBf16 = 1; // matches QSKV_BF16

struct MetaArgs;
struct SelectArgs;
struct DecodeArgs;
struct PrefixArgs;

// Workspace layout: every region starts on a 256-byte boundary.
struct WorkspaceLayout {
    size_t flags;        // uint32 error word (+ padding to 256 B)
    size_t tickets;      // uint32 [rows] per-row counters of the decode's fold (zero between calls)
    size_t scores;       // fp32  [rows][max_pages]
    size_t part_o;       // fp32  [slots][G][D]
    size_t part_lse;     // fp32  [slots][G]
    size_t total;
    int64_t slots;       // rows + decode warps (+ rows x prefix splits)
};

// Decode grid shape on a device with `num_sms` SMs.
struct DecodeGrid {
    int ctas;
    int warps_per_cta;
    int64_t total_warps;
};

DecodeGrid decode_grid(int num_sms, int head_dim);
// L2 bytes of the current device (cached per device; 0 if it cannot be read).
int l2_cache_bytes();
// extra_per_row: partial slots per row for the shared-prefix pieces of a
// cascade decode (0 otherwise).
WorkspaceLayout workspace_layout(int64_t rows, int group, int head_dim, int max_pages, int num_sms,
                                 int extra_per_row = 0);

cudaError_t launch_meta_build(const MetaArgs &a, int kv_dtype, int head_dim, cudaStream_t stream);
// Block Top-K: fp32 mean key per (page, KV head) into a.meta; scores q . centroid.
cudaError_t launch_centroid_build(const MetaArgs &a, int kv_dtype, int head_dim, cudaStream_t stream);
cudaError_t launch_page_select_centroid(const SelectArgs &a, int q_dtype, int head_dim, cudaStream_t stream,
                                        int score_all);
// score_all: compute scores even for rows where every page is kept.
// refresh: recompute each row's last-page metadata from a.k_pool first (bf16 only).
cudaError_t launch_page_select(const SelectArgs &a, int q_dtype, int meta_dtype, int head_dim, cudaStream_t stream,
                               int score_all, int refresh = 0, int rank = 1);
// tmap_k / tmap_v are used by the bf16 tensor-core kernels only.  With
// `prefix` (a cascade decode, bf16 KV) the shared-prefix kernel runs between
// the decode and the merge.
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap *tmap_k, const CUtensorMap *tmap_v, int q_dtype,
                          int kv_dtype, int head_dim, const DecodeGrid &grid, cudaStream_t stream,
                          const PrefixArgs *prefix = nullptr);
// LSE merge of the decode rows split over several warps (and of another
// kernel's extra pieces); launched after the decode grid.
cudaError_t launch_merge(const DecodeArgs &a, int head_dim, cudaStream_t stream);
// Shared-prefix attention of a cascade decode: 128-row query tiles per KV
// head, and the key splits per (tile, head) chosen for a device with
// `num_sms` SMs (0 when the prefix is empty).
int prefix_tiles(int batch, int group);
// Persistent CTAs of the prefix grid for `items` items on a device with `num_sms` SMs.
int prefix_ctas(int items, int num_sms);
int prefix_splits(int batch, int group, int num_kv_heads, int page_size, int prefix_pages, int num_sms);
cudaError_t launch_prefix(const PrefixArgs &a, const CUtensorMap *tmap_k, const CUtensorMap *tmap_v, int q_dtype,
                          int head_dim, cudaStream_t stream);
// Size of the static device scratch used by qskv_sparse_paged_decode_noalloc
// and its device address on the current device (looked up on first use).
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;
cudaError_t noalloc_scratch_address(void **ptr);

// CTAs per row of the one-row-per-CTA decode for `rows` rows of
// slots_per_row units on a grid of `ctas` CTA slots (0: use the stream-K
// split instead).
int row_blocks_for(int64_t rows, int slots_per_row, int ctas, bool no_extra_pieces, bool have_tickets);
// Shared memory the one-row-per-CTA decode needs beyond the rings (the unit
// codes, the page-table row when a.pt_in_smem, the group's queries of
// q_bytes each), and the dynamic shared memory a decode CTA may take with
// two CTAs per SM on the current device.
size_t rowcta_extra_smem(const DecodeArgs &a, int q_bytes);
size_t rowcta_smem_budget();

// Stage count and dynamic shared memory of the bf16 decode kernel.
int decode_stages(int head_dim);
int decode_warps_per_cta(int head_dim);
size_t decode_smem_bytes(int head_dim, int stages);
// Pages one decode CTA can stage for the fused scoring in one round.
int fused_score_pages_per_round(int head_dim);

}  // namespace qskv
