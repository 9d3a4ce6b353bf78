// qh_tmap.h -- host-side TMA tensor-map helpers and tensor-core launchers.
#pragma once

#include <cuda.h>

#include "qh_internal.cuh"

namespace qh {

// fp16 row-major matrix [rows, cols], box of 64 columns x box_rows rows,
// 128-byte swizzle (the tensor core's K-major SW128 layout).
bool tmap_rows_f16_sw128(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                         uint32_t box_rows);

// Packed uint32 head [rows, words_per_row], box of box_words x box_rows, no swizzle.
bool tmap_packed_rows(CUtensorMap* map, const uint32_t* wq, uint64_t words_per_row, uint64_t rows,
                      uint32_t box_words, uint32_t box_rows);

// Same with 128-byte rows in shared memory and the 128-byte swizzle: 16-byte
// chunk j of box row r lands at chunk j ^ (r & 7) (box of 32 words x box_rows;
// the destination must be 1024-byte aligned).
bool tmap_packed_rows_sw128(CUtensorMap* map, const uint32_t* wq, uint64_t words_per_row,
                            uint64_t rows, uint32_t box_rows);

// Packed uint32 head, box of box_words (8, 16 or 32) x box_rows, rows of
// 32, 64 or 128 bytes in shared memory with the swizzle of the same span:
// 16-byte chunk c of box row r lands at c ^ ((r >> 2) & 1) (32 B),
// c ^ ((r >> 1) & 3) (64 B) or c ^ (r & 7) (128 B); the destination must be
// aligned to 256, 512 or 1024 bytes respectively.
bool tmap_packed_rows_swz(CUtensorMap* map, const uint32_t* wq, uint64_t words_per_row,
                          uint64_t rows, uint32_t box_words, uint32_t box_rows);

// Per-group fp16 table [rows, groups] (scales or biases), box of box_groups x
// box_rows, no swizzle.  The row pitch (groups * 2 bytes) must be a multiple
// of 16 bytes and box_groups a multiple of 8; false otherwise.
bool tmap_group_rows(CUtensorMap* map, const void* scales, uint64_t groups, uint64_t rows,
                     uint32_t box_groups, uint32_t box_rows);

// Vocab rows per tile of the tensor-core logit kernel (its MMA N); vocab
// ranges handed to it are counted in these tiles.
constexpr int kTcFwdTileRows = 256;
// Vocab rows of a tile each CTA of the logit kernel's CTA pair loads (the
// packed head's tensor map box height; unswizzled rows of 64 codes).
constexpr int kTcFwdBoxRows = 128;

// Arguments of the tensor-core logit kernel (forward and backward phase 1).
struct TcFwdArgs {
    const __half* scales;
    const __half* biases;
    int64_t V;
    int H;
    float cap;
    const int* count;   // active rows (device)
    int* err;           // error word (device)
    int stall;          // test switch: the producer issues no loads (waits expire)
    int vt_begin, vt_end;  // vocab tiles (kTcFwdTileRows rows) covered by this launch
    // softmax epilogue (forward)
    Partial* part;
    int* S_out;
    // coefficient epilogue (backward phase 1)
    const float* lse;   // [M], original row order
    const int* rows;    // compact -> original row (also for bmax)
    __half* coeff;      // [coeff_rows, coeff_ld]
    int64_t coeff_ld;
    int coeff_rows;
    // blockMax early exit: the forward's per-tile maxima of z (softmax
    // epilogue; [M, bmax_ld], original row order) and the backward's skip map
    // (coefficient epilogue; [128-row tile, skip_ld], 1 = skip the vocab tile)
    float* bmax;
    int64_t bmax_ld;
    const uint8_t* skip;
    int64_t skip_ld;
    int skip_rows;      // 128-row tiles in the skip map
    // Coefficient filter (EPI_FILTER epilogue): a block of 32 compact rows x
    // 32 vocab rows is cold when no row's target lies in it and every
    // p * sech2 * |dlogp| < filter_eps; its coefficients are written as
    // zeros.  A warm block clears bit k & 63 of kbits[u * kbits_ld + k / 64]
    // (256-row dh unit u, 64-row vocab step k of the head); cold_out, when
    // set, gets cold_out[rg * cold_out_ld + vc] = 1 for a cold block (row
    // block rg, vocab block vc < cold_out_ld), 0 for a warm one.
    const float* dlogp;     // [M], original row order
    const int32_t* targets; // [M], original row order
    float filter_eps;
    unsigned long long* kbits;
    int64_t kbits_ld;
    uint8_t* cold_out;
    int64_t cold_out_ld;
    int64_t cold_out_rows;
    // Set by launch_tc_fwd: the scale and bias tables are staged by TMA.
    int sb_tma;
};

// Arguments of the tensor-core dh contraction (backward phase 2).
struct TcDhArgs {
    const __half* scales;
    const __half* biases;
    int64_t V;
    int H;
    const int* count;     // active rows (device)
    int* err;             // error word (device)
    const int* rows;      // compact -> original row
    const float* dlogp;   // [M], original row order
    float* dh_acc;        // [ks][Mpad, H] fp32, compact rows, one buffer per K slice
    int64_t slice_stride; // elements between K-slice buffers (Mpad * H)
    int64_t v_begin;      // first vocab row of the chunk
    int n_k;              // 64-row vocab steps in the chunk
    int ks;               // K slices per output tile (each adds into its own buffer)
    int accumulate;       // 0: write, 1: add to dh_acc
    // blockMax early exit: skip map [skip_rows 128-row tiles, skip_ld vocab
    // tiles of 256 rows]; a K step is skipped when both 128-row tiles of the
    // unit skip its vocab tile (NULL: no skipping)
    const uint8_t* skip;
    int64_t skip_ld;
    int skip_rows;
    // Coefficient filter: bit k & 63 of kbits[unit * kbits_ld + k / 64] set =
    // the unit's 64-row vocab step k of the head (counted from row 0) holds
    // only cold blocks and is skipped (NULL: no skipping)
    const unsigned long long* kbits;
    int64_t kbits_ld;
};

// Arguments of the head-gradient contraction (one vocab chunk).
struct TcDwArgs {
    int64_t V;
    int H;
    const int* count;          // active rows (device)
    int* err;                  // error word (device)
    int stall;                 // test switch: the producer issues no loads (waits expire)
    int64_t v_begin;           // first vocab row of the chunk
    int chunk_rows;            // vocab rows of the chunk (<= the coefficient block's columns)
    const float* dmax;         // max |dlogp| over the active rows (device scalar)
    const int* offs;           // [V + 1] one-hot list offsets
    const int* idx;            // one-hot lists: compact rows, ascending per target
    const float* g;            // [Mpad] dlogp * sech2(target logit) per compact row
    const int* rows;           // compact -> original row
    const __nv_bfloat16* h;    // [M, H] original hidden states
    float* dw;                 // [V, H] output, 32-byte aligned
};

int tc_dh_cols(int H);          // hidden columns per output tile (256 or 128)
int tc_dh_words(int H, int bits);
// True when the dh kernel takes its packed tile as 128-byte-swizzled halves
// (tensor map: tmap_packed_rows_sw128 with 64-row boxes); false: unswizzled
// boxes of tc_dh_words words (tmap_packed_rows).
bool tc_dh_swizzled(int H, int bits);
cudaError_t launch_tc_dh(const CUtensorMap& tmap_c, const CUtensorMap& tmap_w, const TcDhArgs& a,
                         int bits, int grid, cudaStream_t st);

int tc_fwd_smem_bytes(int bits);
int tc_dw_smem_bytes(int H);
// max |dlogp|, the scaled fp16 copy h' and the one-hot terms g, and the
// per-target row lists (counting sort, stable in row order).
cudaError_t launch_dw_prep(const uint32_t* wq, SbView sb,
                           int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                           const int* rows, const int* count, const int32_t* targets,
                           const float* dlogp, int64_t Mpad, float* dmax, __half* hp, float* g,
                           int* cnt, int* offs, int* cursor, int* idx, cudaStream_t st);
cudaError_t launch_tc_dw(const CUtensorMap& tmap_c, const CUtensorMap& tmap_hp, const TcDwArgs& a,
                         int grid, cudaStream_t st);
// Writes NaN to all of dw [V, H] if the error word is set (a wait expired).
cudaError_t launch_dw_poison(const int* err, float* dw, int64_t n, cudaStream_t st);
cudaError_t launch_tc_fwd(const CUtensorMap& tmap_h, const CUtensorMap& tmap_w,
                          const TcFwdArgs& a, int bits, bool coeff_epilogue, int grid,
                          cudaStream_t st);

}  // namespace qh
