// qmm_internal.h -- handle layout, launch plans and the internal launchers
// that the C-ABI layer (qmm_api.cu) calls.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>

#include "qmm.h"

namespace qmm {

constexpr int kMaxGroup = 8;

// Device status-word bits (see qmm_get_status).
constexpr unsigned kStatusTimeoutBit = 1u;
constexpr unsigned kStatusBadExpertBit = 2u;

struct Matrix {
    int fmt = 0;
    int64_t N = 0, K = 0, row_bytes = 0;
    const uint8_t *w = nullptr;
    int device = 0;
    int sm_count = 0;
    // workspace: split-K partials, per-row-slice tickets, status word
    float *ws = nullptr;
    size_t ws_floats = 0;
    unsigned *tickets = nullptr;
    size_t n_tickets = 0;
    unsigned *status = nullptr;
    // Q4_K tensor-core paths: 2-D tensor map over the rows (a CUtensorMap)
    alignas(64) unsigned char tmap[128];
    bool has_tmap = false;
    // one-row decode kernel: the 3-D column view with boxes of tmap3_ks
    // super-blocks (0: not encoded yet)
    alignas(64) unsigned char tmap3[128];
    int tmap3_ks = 0;
    // prefill GEMM: tensor maps over the weight bytes (u8) with boxes of the
    // 16-byte super-block header and of one 32-byte nibble chunk, 256 rows
    alignas(64) unsigned char tmap_hdr[128];
    alignas(64) unsigned char tmap_nib[128];  // Q8_0: 80-byte windows, 256 rows
    bool has_gemm_maps = false;
    // Q8_0 expert GEMV: the rows as u32 words, boxes of one 272-byte slice x 32 rows
    alignas(64) unsigned char tmap_moe[128];
    bool has_moe_map = false;
    // batched GEMV scratch: the K-slice partial sums (grown on demand)
    void *tcb_ws = nullptr;
    size_t tcb_ws_bytes = 0;
    // tcgen05 batched decode: prepared activations, slice partials, tickets
    // (grown on demand), and the tensor map over the prepared activations
    void *tc5_buf = nullptr;
    size_t tc5_bytes = 0;
    alignas(64) unsigned char tc5_tmap_b[128];
    int tc5_nc = 0;
    // prefill split-K scratch: the partial products (grown on demand)
    void *gemm_ws = nullptr;
    size_t gemm_ws_bytes = 0;
    // expert-layer scratch (allocated on first qmm_moe_* call)
    void *moe_ws = nullptr;
    size_t moe_ws_bytes = 0;
    cudaStream_t last_stream = nullptr;
};

// Bytes of one row for a supported format (K already validated).
inline int64_t row_bytes_of(int fmt, int64_t K)
{
    switch (fmt) {
    case QMM_Q4_K: return (K / 256) * 144;
    case QMM_Q5_K: return (K / 256) * 176;
    case QMM_Q6_K: return (K / 256) * 210;
    case QMM_IQ4_NL: return (K / 32) * 18;
    default: return (K / 32) * 34;
    }
}

// The further block formats (formats.cu): Q5_K, Q6_K, IQ4_NL.  Decode GEMV
// for 1..16 activation rows (X rows ldx apart, Y rows ldy apart) and block
// decode to fp32 or bf16 (exactly one of out_f32 / out_bf16).
bool is_extra_format(int fmt);
// Matrices that take the per-group kernels of formats.cu: the further formats,
// and Q8_0 rows whose K is a multiple of 32 but not of 256.
bool uses_fmt_kernels(const Matrix &m);
// Decode GEMV of Q5_K / Q6_K / IQ4_NL (K % 256 == 0) at memory speed
// (formats_fast.cu).
// Rows of activations per pass of the fast kernel for M rows (4, 2 or 1), or
// 0 when it does not take the matrix (format, K, shared memory).
int fmt_fast_rows(const Matrix &m, int M);
size_t fmt_fast_smem(int fmt, int64_t K, int MR);
// n matrices (n > 1 only with M == 1) sharing the M activation rows (ldx
// apart); matrix i's outputs at ys[i], rows ldy apart.  Every output row is
// bitwise the same as from a one-row call.
cudaError_t launch_gemv_fmt_fast(const Matrix *const *ms, int n, const float *x, int64_t ldx,
                                 int M, float *const *ys, int64_t ldy, cudaStream_t s);
cudaError_t launch_gemv_fmt(const Matrix &m, const float *X, int M, int64_t ldx, float *Y,
                            int64_t ldy, cudaStream_t s);
cudaError_t launch_dequant_fmt(const Matrix &m, int64_t row0, int64_t nrows, float *out_f32,
                               uint16_t *out_bf16, cudaStream_t s);

// Kernel launches issued by the library (qmm_launch_count): every launcher
// passes its launch status through counted().
void count_launch();
inline cudaError_t counted(cudaError_t e)
{
    if (e == cudaSuccess)
        count_launch();
    return e;
}

// A kernel's dynamic shared-memory limit raised to at least `bytes` on the
// current device (and, with max_carveout, the whole unified L1/shared array
// preferred for shared memory).  Function attributes persist, so the runtime
// is called only when the recorded limit is lower: setting them on every
// launch cost microseconds of host time per call.
cudaError_t func_smem(const void *func, size_t bytes, bool max_carveout = false);
// Resident blocks per SM of `func` at `threads` and `smem`, remembered per
// (device, function, threads, shared memory).
cudaError_t func_occupancy(const void *func, int threads, size_t smem, int *per_sm);

// Programmatic dependent launch on every kernel unless QMM_PDL=0.
inline bool pdl_enabled()
{
    const char *e = getenv("QMM_PDL");
    return !(e && e[0] == '0');
}

// --------------------------------------------------------------- GEMV plan
// A CTA owns a contiguous range of rows (balanced to within one row) and one
// K-slice of `kchunks` 64-weight chunks.  Its threads form `rg` row teams of
// `kchunks` threads; thread c of a team owns chunk c of the slice (its
// activations stay in registers) and the team walks the rows.  Rows reach
// shared memory in stages of `stage_rows` rows by bulk copies.
struct GemvPlan {
    int kchunks = 0;      // chunks (64 weights) per K-slice = team size
    int ksplit = 1;       // number of K-slices
    int rg = 0;           // row teams per CTA
    int rpg = 0;          // rows per team per stage (1, 2 or 4)
    int stage_rows = 0;   // rg * rpg
    int stages = 0;       // ring depth
    int threads = 0;      // rg * kchunks
    int row_slices = 0;   // number of row ranges
    int64_t slice_bytes = 0;  // bytes of one row within one K-slice
    size_t smem = 0;
};

struct GemvArgs {
    int fmt;
    int nmat;                       // matrices sharing x (1 for plain GEMV)
    const uint8_t *w[kMaxGroup];
    float *y[kMaxGroup];
    int64_t row_end[kMaxGroup];     // cumulative row counts
    int64_t N;                      // total rows
    int64_t K;
    int64_t row_bytes;
    const float *x;
    float *ws;                      // [ksplit][N] partials (ksplit > 1)
    unsigned *tickets;              // [row_slices] (ksplit > 1)
    unsigned *status;
};

// Plan for N total rows of K columns; `force_ksplit` > 0 overrides split-K.
GemvPlan plan_gemv(int fmt, int64_t N, int64_t K, int sm_count, int force_ksplit);
size_t gemv_workspace_floats(const GemvPlan &p, int64_t N);
// Whether launch_gemv takes this plan for the format (Q5_K / Q6_K / IQ4_NL
// need 32-lane teams and 16-byte row and slice sizes).
bool gemv_plan_takes(int fmt, const GemvPlan &p, int64_t row_bytes);
cudaError_t launch_gemv(const GemvPlan &p, const GemvArgs &a, cudaStream_t s);

// --------------------------------------------------------------- tensor-core Q4_K GEMV
struct TcArgs {
    const void *tmap[kMaxGroup];  // 128-byte CUtensorMap of each matrix
    int64_t rows[kMaxGroup];
    float *y[kMaxGroup];
    int nmat;
    int64_t K;
    int M;                // activation rows, 1..4
    int64_t ldx, ldy;     // row strides of X and Y (elements)
    const float *x;
    unsigned *status;
    int fuse_swiglu;      // nmat == 2, M == 1, equal shapes: y[0] = silu(m0 x) * (m1 x)
};
size_t gemv_tc_smem(int64_t K, int M, int nslot, int nw, int res_tiles = 0);
cudaError_t launch_gemv_tc(const TcArgs &a, int sm_count, cudaStream_t s);
int make_q4k_tensor_map(void *out128, const void *w, int64_t N, int64_t row_bytes);

// --------------------------------------------------------------- one-row Q4_K decode GEMV
// gemv_m1.cu: a producer warp streams 16-row units into a shared-memory ring,
// one consumer warp per super-block of a K slice runs the tensor-core unit;
// work items (tile groups) are handed out first statically, then from a
// counter per slice.
constexpr int kM1MaxWarps = 16;
constexpr size_t kM1SmemBudgetWhole = 226 * 1024;  // one CTA per SM
constexpr size_t kM1SmemBudgetHalf = 110 * 1024;   // two CTAs per SM
struct M1Plan {
    int maxw = 0;                // consumer warps at most: 8 (half an SM) or 16
    int S = 0, KS = 0;           // K slices, super-blocks per slice
    int WS = 0, NP = 0;          // super-blocks per pass, passes per item (KS = WS * NP)
    int TS = 0, W = 0;           // tiles per item, consumer warps (WS * TS / upw)
    int upw = 1;                 // units per consumer warp and slot
    int G1 = 0;                  // CTAs per slice (grid = G1 * S)
    int n_items = 0;             // items per slice
    int F = 0;                   // fixed items per CTA (fetched before the PDL wait)
    int cap = 0;                 // items a CTA may take
    int nslot = 0, slot_bytes = 0;
    size_t smem = 0;
    size_t ws_floats = 0;        // K-slice partial sums (S > 1)
    size_t tickets = 0;          // counters: 2 per slice, plus one per item when S > 1
};
struct M1Args {
    int fmt;                      // QMM_Q4_K or QMM_Q5_K
    const void *tmap[kMaxGroup];  // Matrix::tmap3 of each matrix (boxes of WS super-blocks)
    int64_t rows[kMaxGroup];
    float *y[kMaxGroup];
    int nmat;
    const float *x;
    float *ws;
    unsigned *tickets;
    unsigned *status;
    int fuse_swiglu;              // nmat == 2 (gate, up of equal rows): y[0] = silu(gate) * up
};
// T: 16-row tiles over all matrices; NB: super-blocks per row; force_S > 0
// fixes the number of K slices (it must divide NB).
// maxw: 8 or 16 consumer warps at most (0: QMM_M1_WARPS, default 16).
// nslot == 0: no plan fits.
// sb_bytes: 144 (Q4_K) or 176 (Q5_K).
// min_ts: the least tiles per item (2 for the fused gate/up pairs); upw:
// units per consumer warp and ring slot (1, or 2: W = WS * TS / 2).
M1Plan plan_m1(int64_t T, int64_t NB, int sm_count, int force_S, int maxw = 0,
               int sb_bytes = 144, int min_ts = 1, int upw = 1);
size_t m1_smem(int KS, int WS, int TS, int cap, int nslot, int sb_bytes = 144);
cudaError_t launch_gemv_m1(const M1Args &a, const M1Plan &p, cudaStream_t s);

// --------------------------------------------------------------- batched tensor-core Q4_K GEMV
// Up to 16 activation rows in one pass; CTA (r, s) of an R x S grid owns a
// range of row tiles and a slice of K (see gemv_batched.cu).
struct TcbPlan {
    int nt = 0;            // groups of four activation rows
    int S = 0, R = 0;      // K slices, row groups (S == 0: does not fit)
    int kc = 0;            // super-blocks per slice (at most)
    size_t smem = 0;
    size_t ws_floats = 0;  // partial sums, S * M * N when S > 1
    size_t tickets = 0;    // row-group tickets: R when the slices are added in-kernel, else 0
};
struct TcbArgs {
    const void *tmap;      // Matrix::tmap
    const float *x;
    float *y;
    float *ws;             // plan.ws_floats floats when S > 1
    unsigned *tickets;     // plan.tickets zeroed counters (reset by the kernel)
    unsigned *status;
    int64_t ldx, ldy, N, K;
    int M;
};
TcbPlan plan_tcb(int64_t N, int64_t K, int M, int sm_count);
cudaError_t launch_gemv_tcb(const TcbArgs &a, const TcbPlan &p, cudaStream_t s);

// --------------------------------------------------------------- TMA tensor maps
// Encode a 2-D tiled tensor map (dtype: a CUtensorMapDataType, swizzle: a
// CUtensorMapSwizzle); 0 on success.
int encode_tmap_2d(void *out128, int dtype, const void *base, uint64_t dim0, uint64_t dim1,
                   uint64_t stride1_bytes, uint32_t box0, uint32_t box1, int swizzle);
// The same for a 3-D tensor (dims innermost first, strides of dims 1 and 2).
int encode_tmap_3d(void *out128, int dtype, const void *base, uint64_t dim0, uint64_t dim1,
                   uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                   uint32_t box1, uint32_t box2, int swizzle);
// 3-D column view (super-block bytes as u64 words, row, super-block) with
// boxes of 16 rows x ks super-blocks; sb_bytes 144 (Q4_K) or 176 (Q5_K).
int make_column_map(void *out128, const void *w, int64_t N, int64_t row_bytes, int ks,
                    int sb_bytes);

// --------------------------------------------------------------- prefill GEMM
constexpr int kGemmMaxGroup = 4;
struct GemmArgs {
    int fmt;                             // QMM_Q4_K or QMM_Q8_0
    const void *tmap_x;                  // X [M][K] bf16: box 64 x tok, 128-byte swizzle
    const void *tmap_hdr[kGemmMaxGroup]; // Matrix::tmap_hdr of each matrix
    const void *tmap_nib[kGemmMaxGroup]; // Matrix::tmap_nib
    float *y[kGemmMaxGroup];             // [M][N_i]
    int64_t N[kGemmMaxGroup];
    int nmat;
    float *ws;             // split-K partials (gemm_q4k_ws_floats floats) when ksplit > 1
    int ksplit;            // K slices of each tail tile
    int full_tiles;        // tiles that run whole (the rest are split) when ksplit > 1
    int tok;               // token tile height: 256, or 128 when 256-token tiles are too few
    int64_t M, K;
    unsigned *status;
};
size_t gemm_q4k_smem(int tok, int fmt);
int gemm_q4k_tiles(int64_t M, int64_t N, int tok);
struct GemmSplit {
    int full;    // whole tiles (the first ones)
    int ksplit;  // K slices of each remaining tile (1: none split)
};
GemmSplit gemm_q4k_split(int tiles, int tok, int64_t K, int sm_count);
size_t gemm_q4k_ws_floats(int64_t M, int64_t Ntot, int ksplit);
cudaError_t launch_gemm_q4k(const GemmArgs &a, int sm_count, cudaStream_t s);

// --------------------------------------------------------------- mixture of experts
// Slots of one expert are processed in groups of at most kGroupTokens tokens
// (the activation rows of one tensor-core pass).
constexpr int kGroupTokens = 4;
constexpr int kMoeMaxSlots = 4096;   // T * top_k
constexpr int kMoeMaxExperts = 512;
constexpr int kMoeMaxTopK = 16;

// The bucketing result on the device.
struct MoeIndex {
    int4 *groups;   // [<= S / kGroupTokens + E] {expert, first, count, 0}
    int *slots;     // [S] slots sorted by (expert, slot)
    int *n_groups;  // [1]
};
inline size_t moe_max_groups(int S, int E) { return size_t(S / kGroupTokens + E); }

struct MoeExpertArgs {
    const void *tmap[2];  // stacked expert matrices (n_experts * Ne rows each)
    float *y[2];          // per-slot outputs, [S][Ne]
    int nmat;             // 1, or 2 for gate and up together
    int64_t Ne, K;
    const float *x;
    int64_t ldx;
    int top_k;
    int x_per_slot;
    const float *xscale;  // per-slot input scale [T*top_k] (routing on the input), or null
    int fuse_swiglu;      // nmat == 2: y[0] = silu(gate) * up, y[1] unused
    int maxpairs;         // (fused) shared-memory room: (gate, up) tile pairs per CTA
    MoeIndex ix;
    unsigned *status;
};

size_t moe_bucket_smem(int S, int E);
cudaError_t launch_moe_bucket(const int32_t *ids, int S, int E, const MoeIndex &ix, float *y0,
                              int64_t n0, int64_t ld0, unsigned *status, cudaStream_t s);
void moe_expert_shape(int64_t K, int &nw, int &nslot);
size_t moe_expert_smem(int64_t K, int nw, int nslot, int maxpairs);
cudaError_t launch_moe_expert(const MoeExpertArgs &a, int sm_count, cudaStream_t s);
// moe_q8.cu: the expert GEMV for Q8_0 weights (K % 256 == 0), on the same
// bucketing and arguments (tmap: the maps of encode_moe_q8_map; maxpairs
// unused; SwiGLU fusion always fits).
int moe_q8_sps(int64_t NB);     // K-slices per stage (1 or 2)
size_t moe_q8_smem(int sps);
int encode_moe_q8_map(void *out128, const void *w, int64_t N, int64_t row_bytes);
cudaError_t launch_moe_q8(const MoeExpertArgs &a, int sm_count, cudaStream_t s);
cudaError_t launch_swiglu(const float *g, const float *u, float *h, int64_t n, int sm_count,
                          cudaStream_t s);
cudaError_t launch_moe_combine(const float *ys, const float *r, const int32_t *ids, int E, int T,
                               int top_k, int64_t Ne, float *y, int sm_count, cudaStream_t s);

// --------------------------------------------------------------- batched decode on tcgen05
// gemv_tc5.cu: Q4_K, 2..16 activation rows, 256-row tiles x K slices.
struct Tc5Plan {
    int nc = 0;             // B columns: 16 (T <= 8) or 32 (T <= 16)
    int tiles = 0;          // 256-row tiles
    int S = 1, sbs = 0;     // K slices, super-blocks per slice
    int items = 0;          // tiles * S
    size_t smem = 0;
    size_t ws_floats = 0;   // slice partials [S][tiles][256][16] (S > 1)
    size_t tickets = 0;     // [tiles][8]
    size_t prep_bytes = 0;  // prepared activations: [nc][K] f16, scales, sub-block sums
};
Tc5Plan plan_tc5(int64_t N, int64_t K, int T, int sm_count);
struct Tc5Args {
    const void *tmap_hdr, *tmap_nib;  // Matrix::tmap_hdr / tmap_nib
    const void *tmap_b;               // the prepared activations: [nc][K] f16, box 64 x nc, SW128
    void *prep;                       // plan.prep_bytes
    float *ws;                        // plan.ws_floats
    unsigned *tickets;                // plan.tickets, zeroed once
    const float *X;
    int64_t ldx;
    float *Y;
    int64_t ldy;
    int64_t N, K;
    int T;
    unsigned *status;
};
cudaError_t launch_gemv_tc5(const Tc5Plan &p, const Tc5Args &a, int sm_count, cudaStream_t s);

// --------------------------------------------------------------- Q8_K integer-dot path
struct Q8kArgs {
    const uint8_t *w[kMaxGroup];  // Q4_K matrices sharing K
    float *y[kMaxGroup];
    int64_t N[kMaxGroup];
    int nmat;
    int64_t K;
    const uint8_t *xq;            // Q8_K blocks of the activations (K/256 x 292 bytes)
    const float *x;               // or (non-null) the f32 activations, quantized in the GEMV
};
size_t q8k_smem(int64_t K);
cudaError_t launch_quantize_q8k(const float *x, int64_t K, uint8_t *out, cudaStream_t s);
cudaError_t launch_gemv_q8k(const Q8kArgs &a, int sm_count, cudaStream_t s);

// --------------------------------------------------------------- no-allocation entry
// Layout of qmm_gemv_noalloc's static scratch: [status word, padded to 256 B]
// [tickets][split-K partial sums], 1 MiB in total.
constexpr size_t kNoallocScratchBytes = size_t(1) << 20;
constexpr size_t kNoallocStatusBytes = 256;
constexpr size_t kNoallocTickets = 4096;
constexpr size_t kNoallocPartialFloats =
    (kNoallocScratchBytes - kNoallocStatusBytes - kNoallocTickets * 4) / 4;

// Whether a decode GEMV plan's split-K scratch fits the static array.
inline bool noalloc_fits(const GemvPlan &p, int64_t N)
{
    return gemv_workspace_floats(p, N) <= kNoallocPartialFloats &&
           size_t(p.row_slices) <= kNoallocTickets;
}

// Argument checks of qmm_gemv_noalloc, and recording its refusal sentence for
// qmm_last_error().
qmm_status noalloc_check(int fmt, int64_t N, int64_t K, const void *w, const float *x,
                         const float *y);
qmm_status noalloc_fail(qmm_status code, const char *fmt, ...);

// --------------------------------------------------------------- dequant
cudaError_t launch_dequant(const Matrix &m, int64_t row0, int64_t nrows, float *out_f32,
                           uint16_t *out_bf16, cudaStream_t s);

} // namespace qmm
