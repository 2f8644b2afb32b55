// gemv_tc.cu -- Q4_K decode GEMV (M = 1..4 activation rows) on the tensor
// cores, with the dequantisation fused into the operand construction.
//
// The operation: "Building a Rust Inference Engine That Matches Llama.cpp",
// "Where the wins came from" -- the dequant math happens inline in the dot
// product; the weights never become a full-precision buffer.
//
// Why tensor cores for a GEMV.  Decoding Q4_K in plain fp32 costs one
// integer-pipe instruction per weight (isolate the nibble) plus an FMA, and
// the integer pipe (16 lanes per scheduler) then caps the kernel below the
// HBM rate.  Here two nibbles are isolated per instruction straight into an
// fp16 pair, and mma.sync multiplies them by the activations.  The
// activations enter as two fp16 terms (hi + lo, about 22 significant bits)
// after an exact power-of-two scale per super-block, so the products are
// exact and only the fp32 accumulation rounds.
//
// One activation row (the decode case): the nibbles enter unscaled, as fp16
// subnormals (w & 0x000F000F is the half2 (q0, q1) * 2^-24), and each pair of
// MMA columns collects one sub-block (hi and lo activation terms), so the
// scales and mins apply once per sub-block in fp32 (tc_common.cuh,
// unit_dot_sb).  Two to four rows: one
// exact fp16 FMA, (1024+q)*sc - 1024*sc = q*sc (<= 945, exact in fp16), on
// (w & 0x000F000F) | 0x64006400 applies the sub-block scale to the operand,
// and the mins are a second small MMA per super-block (m_s against the
// sub-block sums of x, scaled by a further 2^-5 to stay inside fp16).  Per
// super-block and row: y += (d*Dq - dmin*32*Dmin) * 2^-s.
//
// Work decomposition.  The matrix is cut into units of 16 rows x one
// 256-weight super-block column (2304 bytes), ordered (matrix, row tile,
// super-block).  Every CTA owns whole row tiles (an even split, so CTAs
// differ by at most one tile) and splits their units evenly over its warps.
// A warp streams its units through its own ring of shared-memory slots with
// 2-D TMA copies (no CTA-wide synchronisation in the loop), keeps its rows'
// partial sums in registers, and writes a row tile directly when it covered
// the whole tile.  Tiles split between warps are added in shared memory at the
// end, in warp order: no global synchronisation, and results are bitwise
// repeatable.
//
// Fragment layout (mma.sync m16n8k16, A row-major, B col-major): lane = 4g+c.
// (Two to four activation rows; the one-row layout is described with
// unit_dot_sb.)
// For a 16-row tile, lane (g, c) holds rows g and g+8 and owns chunk c of the
// super-block (qs bytes 32c..32c+31: sub-blocks 2c and 2c+1).  Word t of the
// chunk feeds k-steps 2t and 2t+1: step 2t takes nibbles (0,4) [sub-block 2c]
// in k-slots (2c, 2c+1) and nibbles (1,5) [sub-block 2c+1] in (2c+8, 2c+9);
// step 2t+1 takes nibbles (2,6) and (3,7).  The B fragment for the same
// (step, c) holds the matching activations; column n of B is (x row n/2,
// term n%2), so lane c's accumulator columns (2c, 2c+1) are both terms of
// activation row c.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cuda.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "tc_common.cuh"

namespace qmm {

namespace {

using namespace tc;

struct TcParams {
    CUtensorMap tmap[kMaxGroup];  // rows of each matrix as a 2-D uint64 tensor
    int64_t tile_end[kMaxGroup];  // cumulative 16-row tile counts
    int64_t rows[kMaxGroup];
    float *y[kMaxGroup];
    const float *x;
    unsigned *status;
    int64_t U;          // units
    int64_t ldx, ldy;   // activation / output row strides (elements)
    int nmat, M, NB, nslot;
    int late_trigger;           // let the next kernel launch only after the main loop
    // fuse = 1 (two matrices of the same shape, M = 1): tiles are taken as
    // (gate, up) pairs of the same rows, staged in shared memory (room for
    // res_tiles tiles per CTA), and y[0] receives h = silu(gate x) * (up x).
    int fuse;
    int res_tiles;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

__device__ __forceinline__ int matrix_of_tile(const TcParams &P, int64_t tile)
{
    int m = 0;
#pragma unroll
    for (int i = 0; i < kMaxGroup - 1; ++i)
        if (i < P.nmat - 1 && tile >= P.tile_end[i])
            m = i + 1;
    return m;
}

// A position in the unit sequence, advanced without divisions.
struct Cursor {
    int tile;     // global 16-row tile
    int sb;       // super-block column
    int mat;      // matrix of the tile
    int tend;     // first global tile of the next matrix
    int tbase;    // first global tile of this matrix
};

__device__ __forceinline__ Cursor cursor_at(const TcParams &P, int64_t u)
{
    Cursor q;
    q.tile = int(u / P.NB);
    q.sb = int(u % P.NB);
    if (P.fuse) {
        q.mat = q.tile & 1;
        q.tbase = q.tile - (q.tile >> 1);  // so that tile - tbase = the row tile
        q.tend = 0;
        return q;
    }
    q.mat = matrix_of_tile(P, q.tile);
    q.tbase = q.mat == 0 ? 0 : int(P.tile_end[q.mat - 1]);
    q.tend = int(P.tile_end[q.mat]);
    return q;
}

__device__ __forceinline__ void advance(const TcParams &P, Cursor &q)
{
    if (++q.sb == P.NB) {
        q.sb = 0;
        ++q.tile;
        if (P.fuse) {
            q.mat = q.tile & 1;
            q.tbase = q.tile - (q.tile >> 1);
        } else if (q.tile == q.tend && q.mat + 1 < P.nmat) {
            ++q.mat;
            q.tbase = q.tend;
            q.tend = int(P.tile_end[q.mat]);
        }
    }
}

template <int NCOL>
__global__ void __launch_bounds__(512, 1) gemv_tc_kernel(const __grid_constant__ TcParams P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int nw = int(blockDim.x) >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int NB = P.NB, M = P.M, NS = P.nslot;

    uint8_t *ring = smem + size_t(warp) * NS * kTileBytes;
    uint8_t *acts = smem + size_t(nw) * NS * kTileBytes;
    // One activation row (NCOL == 2): the per-sub-block B layout of
    // tc_common.cuh, Bx [NB][16][4][2] uint2, its zero block Zx [16][8] and
    // the sub-block sums Xs [NB][8].  Several rows: Bs [NB][16][NCOL][4] and
    // the min-MMA fragments Bm [NB][NCOL][4].
    uint2 *Bx = reinterpret_cast<uint2 *>(acts);
    uint2 *Zx = Bx + size_t(NB) * 128;
    float *Xs = reinterpret_cast<float *>(Zx + 128);
    uint2 *Bs = reinterpret_cast<uint2 *>(acts);
    uint32_t *Bm = reinterpret_cast<uint32_t *>(Bs + size_t(NB) * 16 * NCOL * 4);
    float *inv = NCOL == 2 ? Xs + size_t(NB) * 8
                           : reinterpret_cast<float *>(Bm + size_t(NB) * NCOL * 4);  // [NB][M]
    float *part = inv + size_t(NB) * M;                                              // [nw][2][4][16]
    float *res = part + size_t(nw) * 2 * 4 * kTileRows;  // fused: [res_tiles][16] tile results
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(res + size_t(P.fuse ? P.res_tiles : 0) * kTileRows) + 7) &
        ~uintptr_t(7));
    uint64_t *bar = bars + warp * NS;

    // Each CTA owns whole row tiles (split evenly, G <= tiles) and splits
    // their units evenly over its warps.
    const int64_t G = gridDim.x;
    const int64_t T = P.U / NB;
    // Fused: whole (gate, up) pairs per CTA.
    const int64_t tu = P.fuse ? 2 : 1;
    const int64_t cU0 = (blockIdx.x * (T / tu) / G) * tu * NB,
                  cU1 = ((blockIdx.x + 1) * (T / tu) / G) * tu * NB;
    const int64_t cn = cU1 - cU0;
    auto warp_begin = [&](int w) { return cU0 + int64_t(w) * cn / nw; };
    const int64_t u0 = warp_begin(warp), u1 = warp_begin(warp + 1);
    const int nu = int(u1 - u0);
    __shared__ int wbeg[17];  // warp boundaries relative to cU0 (wbeg[nw] = cn)
    if (lane == 0) {
        wbeg[warp] = int(u0 - cU0);
        if (warp == nw - 1)
            wbeg[nw] = int(cn);
    }

    if (lane == 0) {
        for (int s = 0; s < NS; ++s)
            mbar_init(&bar[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (!P.late_trigger)
        pdl_launch_dependents();

    uint64_t policy = 0;
    Cursor qi = cursor_at(P, u0);  // next unit to request
    int slot_i = 0;
    auto issue = [&]() {
        mbar_arrive_expect_tx(&bar[slot_i], kTileBytes);
        tma_load_2d(ring + size_t(slot_i) * kTileBytes, &P.tmap[qi.mat], qi.sb * 18,
                    (qi.tile - qi.tbase) * kTileRows, &bar[slot_i], policy);
        advance(P, qi);
        if (++slot_i == NS)
            slot_i = 0;
    };
    // Weights are constant: start streaming before waiting for the previous
    // kernel in the stream.
    int issued = nu < NS ? nu : NS;
    if (lane == 0) {
        policy = policy_evict_first();
        for (int j = 0; j < issued; ++j)
            issue();
    }

    pdl_wait();  // x, y and the workspace belong to the previous kernel until here

    // ---- activations -> B fragments.  Warp w takes super-blocks w, w+nw, ...;
    // the loads of up to 8 of them are in flight together.
    {
        const int cc = lane >> 3, tt = lane & 7;
        for (int m = 0; m < M; ++m) {
            for (int sb0 = warp; sb0 < NB; sb0 += 8 * nw) {
                float4 v[8], w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int sb = sb0 + i * nw;
                    if (sb < NB) {
                        const float *xr =
                            P.x + int64_t(m) * P.ldx + int64_t(sb) * 256 + 64 * cc + 4 * tt;
                        v[i] = __ldg(reinterpret_cast<const float4 *>(xr));
                        w[i] = __ldg(reinterpret_cast<const float4 *>(xr + 32));
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int sb = sb0 + i * nw;
                    if (sb < NB) {
                        if constexpr (NCOL == 2)
                            prep_super_block_sb(sb, v[i], w[i], lane, Bx, Xs, inv);
                        else
                            prep_super_block<NCOL>(sb, m, M, v[i], w[i], lane, Bs, Bm, inv);
                    }
                }
            }
        }
        if constexpr (NCOL == 2)
            for (int i = threadIdx.x; i < 128; i += blockDim.x)
                Zx[i] = make_uint2(0u, 0u);
    }
    __syncthreads();

    // ---- main loop
    uint32_t selA, selB;
    bool hi4;
    chunk_selectors(c, selA, selB, hi4);
    const int col = g % NCOL;  // columns beyond 2M repeat real ones (finite, never stored)
    const int mrow = c;        // activation row whose two terms sit in this lane's columns
    const int minv = mrow < M ? mrow : 0;
    const uint8_t *rowA = ring + g * 144;
    // NCOL == 2: lanes g = 2c and 2c+1 read their half of the chunk's B entry,
    // the others the zero block.
    const bool bact = (g >> 1) == c;
    const int boff = 2 * c + (g & 1);
    float *mypart = part + size_t(warp) * 2 * 4 * kTileRows;
    float tot0 = 0.f, tot1 = 0.f;
    Cursor q = cursor_at(P, u0);
    int slot = 0;
    unsigned parity = 0;
    int jfail = -1;

    for (int j = 0; j < nu; ++j) {
        if (!mbar_wait_bounded(&bar[slot], parity)) {
            jfail = j;
            break;
        }
        if constexpr (NCOL == 2) {
            const uint2 *bx = bact ? Bx + (size_t(q.sb) * 128 + boff) : Zx;
            const float2 xab = *reinterpret_cast<const float2 *>(Xs + q.sb * 8 + 2 * c);
            unit_dot_sb(rowA + slot * kTileBytes, c, selA, selB, hi4, bx, xab, inv[q.sb], tot0,
                        tot1);
        } else {
            unit_dot<NCOL>(rowA + slot * kTileBytes, c, selA, selB, hi4,
                           Bs + (size_t(q.sb) * 16 * NCOL + col) * 4 + c,
                           Bm[(size_t(q.sb) * NCOL + col) * 4 + c], inv[q.sb * M + minv], tot0,
                           tot1);
        }

        // Refill this slot with the unit NS ahead: every lane has consumed its
        // loads of the slot (the values fed the MMAs above), so the copy may
        // overwrite it.
        __syncwarp();
        if (issued < nu) {
            if (lane == 0)
                issue();
            ++issued;
        }
        if (++slot == NS) {
            slot = 0;
            parity ^= 1u;
        }

        // ---- the tile ends here (or this warp's share does)
        if (q.sb == NB - 1 || j == nu - 1) {
            if constexpr (NCOL == 2) {
                // The four lanes of a row pair hold two sub-blocks each.
                tot0 += __shfl_xor_sync(0xffffffffu, tot0, 1);
                tot1 += __shfl_xor_sync(0xffffffffu, tot1, 1);
                tot0 += __shfl_xor_sync(0xffffffffu, tot0, 2);
                tot1 += __shfl_xor_sync(0xffffffffu, tot1, 2);
            }
            const int64_t first = int64_t(q.tile) * NB, last = first + NB - 1;
            if (u0 <= first && u1 - 1 >= last) {
                if (P.fuse) {
                    if (mrow == 0) {
                        float *rr = res + (int64_t(q.tile) - cU0 / NB) * kTileRows;
                        rr[g] = tot0;
                        rr[g + 8] = tot1;
                    }
                } else if (mrow < M) {
                    const int64_t rA = int64_t(q.tile - q.tbase) * kTileRows + g;
                    float *yr = P.y[q.mat] + int64_t(mrow) * P.ldy;
                    if (rA < P.rows[q.mat])
                        yr[rA] = tot0;
                    if (rA + 8 < P.rows[q.mat])
                        yr[rA + 8] = tot1;
                }
            } else {
                // Shared with other warps: park this warp's share in shared memory.
                const int k = (u0 >= int64_t(q.tile) * NB) ? 0 : 1;  // first or last tile of this warp
                mypart[(k * 4 + mrow) * kTileRows + g] = tot0;
                mypart[(k * 4 + mrow) * kTileRows + g + 8] = tot1;
            }
            tot0 = tot1 = 0.f;
        }
        advance(P, q);
    }
    if (jfail >= 0) {
        if (lane == 0)
            atomicOr(P.status, kStatusTimeoutBit);
        // Let this warp's copies in flight (units jfail .. issued-1) land
        // before shared memory is released.
        if (lane == 0)
            for (int j = jfail; j < issued; ++j)
                mbar_wait_bounded(&bar[j % NS], unsigned(j / NS) & 1u, 100000000ll);
    }
    if (P.late_trigger)
        pdl_launch_dependents();
    __syncthreads();

    // ---- tiles no single warp covered: add the warps' shares in warp order.
    // Units are counted from the CTA's first one here (32-bit, no divisions
    // inside the loops); warp w owns [wb[w], wb[w+1]).
    const int cm = lane >> 3, cr = lane & 7;  // this lane: x row cm, rows cr and cr+8
    const int ntile = int(cn / NB);
    for (int tr = warp; tr < ntile; tr += nw) {
        const int first = tr * NB, last = first + NB - 1;
        int wf = 0, wl = 0;
        for (int w = 0; w < nw; ++w) {
            const int b0 = wbeg[w];
            if (b0 <= first)
                wf = w;
            if (b0 <= last)
                wl = w;
        }
        if (wf == wl)
            continue;  // written by its warp
        float s0 = 0.f, s1 = 0.f;
        for (int w = wf; w <= wl; ++w) {
            const int b0 = wbeg[w], b1 = wbeg[w + 1];
            if (b1 == b0)
                continue;  // a warp without units
            const int kw = (b0 >= first) ? 0 : 1;  // this tile is w's first (0) or last (1)
            const float *pw = part + (size_t(w) * 2 + kw) * 4 * kTileRows + cm * kTileRows;
            s0 += pw[cr];
            s1 += pw[cr + 8];
        }
        if (P.fuse) {
            if (cm == 0) {
                res[tr * kTileRows + cr] = s0;
                res[tr * kTileRows + cr + 8] = s1;
            }
        } else if (cm < M) {
            const int64_t t = cU0 / NB + tr;
            const int mi = matrix_of_tile(P, t);
            const int64_t rA = (t - (mi == 0 ? 0 : P.tile_end[mi - 1])) * kTileRows + cr;
            float *yr = P.y[mi] + int64_t(cm) * P.ldy;
            if (rA < P.rows[mi])
                yr[rA] = s0;
            if (rA + 8 < P.rows[mi])
                yr[rA + 8] = s1;
        }
    }
    if (!P.fuse)
        return;
    // ---- h = silu(gate) * up for the CTA's (gate, up) tile pairs
    __syncthreads();
    const int npair = ntile / 2;
    const int64_t rt0 = cU0 / NB / 2;  // first row tile of the CTA
    for (int i = threadIdx.x; i < npair * kTileRows; i += blockDim.x) {
        const int pl = i / kTileRows, r = i % kTileRows;
        const int64_t row = (rt0 + pl) * kTileRows + r;
        if (row < P.rows[0])
            P.y[0][row] = silu(res[(2 * pl) * kTileRows + r]) * res[(2 * pl + 1) * kTileRows + r];
    }
}

using TcKernel = void (*)(TcParams);

TcKernel pick_tc(int ncol)
{
    switch (ncol) {
    case 2: return gemv_tc_kernel<2>;
    case 4: return gemv_tc_kernel<4>;
    case 6: return gemv_tc_kernel<6>;
    default: return gemv_tc_kernel<8>;
    }
}

} // namespace

// Warps per CTA and ring depth: 16 warps x 2 slots, the fastest setting of
// a sweep over the Llama-3.1-8B decode step (warps 8-16 x slots 2-6, for
// launches with at least 64 units per CTA -- "big" -- and the rest separately:
// every CTA wants all 16 warps, and deeper rings only add queueing).
// QMM_TC_BIG / QMM_TC_SMALL ("warps,slots") override one class,
// QMM_TC_WARPS / QMM_TC_NSLOT both.
void gemv_tc_shape(int64_t units_per_cta, int &warps, int &nslot)
{
    const bool big = units_per_cta >= 64;
    warps = 16;
    nslot = 2;
    if (const char *c = getenv(big ? "QMM_TC_BIG" : "QMM_TC_SMALL")) {
        int w = 0, n = 0;
        if (sscanf(c, "%d,%d", &w, &n) == 2 && w >= 4 && w <= 16 && n >= 2 && n <= 16) {
            warps = w;
            nslot = n;
        }
    }
    const char *e = getenv("QMM_TC_WARPS");
    if (e && atoi(e) >= 4 && atoi(e) <= 16)
        warps = atoi(e);
    const char *n = getenv("QMM_TC_NSLOT");
    if (n && atoi(n) >= 2 && atoi(n) <= 16)
        nslot = atoi(n);
}

size_t gemv_tc_smem(int64_t K, int M, int nslot, int nw, int res_tiles)
{
    const size_t NB = size_t(K / 256);
    const size_t ncol = 2 * size_t(M);
    const size_t acts = M == 1 ? NB * 128 * 8 + 128 * 8 + NB * 8 * 4 + NB * 4
                               : NB * 16 * ncol * 4 * 8 + NB * ncol * 4 * 4 + NB * M * 4;
    return size_t(nw) * nslot * kTileBytes + acts + size_t(nw) * 2 * 4 * kTileRows * 4 +
           size_t(res_tiles) * kTileRows * 4 + 8 + size_t(nw) * nslot * 8;
}


cudaError_t launch_gemv_tc(const TcArgs &a, int sm_count, cudaStream_t s)
{
    TcParams P;
    memset(&P, 0, sizeof(P));
    int64_t tiles = 0;
    for (int i = 0; i < a.nmat; ++i) {
        P.tmap[i] = *reinterpret_cast<const CUtensorMap *>(a.tmap[i]);
        tiles += (a.rows[i] + kTileRows - 1) / kTileRows;
        P.tile_end[i] = tiles;
        P.rows[i] = a.rows[i];
        P.y[i] = a.y[i];
    }
    for (int i = a.nmat; i < kMaxGroup; ++i)
        P.tile_end[i] = tiles;
    P.x = a.x;
    P.status = a.status;
    P.NB = int(a.K / 256);
    P.U = tiles * P.NB;
    P.ldx = a.ldx;
    P.ldy = a.ldy;
    P.nmat = a.nmat;
    P.M = a.M;
    const char *lt = getenv("QMM_PDL_TRIGGER");
    P.late_trigger = (lt && strcmp(lt, "late") == 0) ? 1 : 0;
    P.fuse = a.fuse_swiglu;
    int64_t ctas = sm_count;
    const int64_t owned = P.fuse ? tiles / 2 : tiles;  // row tiles, or (gate, up) pairs
    if (ctas > owned)
        ctas = owned;  // every CTA owns at least one
    int nw, nslot;
    gemv_tc_shape(P.U / ctas, nw, nslot);
    P.nslot = nslot;
    if (P.fuse)
        P.res_tiles = int(2 * ((tiles / 2 + ctas - 1) / ctas));
    const size_t smem = gemv_tc_smem(a.K, a.M, nslot, nw, P.res_tiles);
    TcKernel kern = pick_tc(2 * a.M);
    cudaError_t e = func_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(unsigned(nw * 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return counted(cudaLaunchKernelEx(&cfg, kern, P));
}

// Describe the rows of a Q4_K matrix as a 2-D tensor of 8-byte elements
// (row_bytes/8 x N) whose boxes are one super-block column of 16 rows.
int make_q4k_tensor_map(void *out128, const void *w, int64_t N, int64_t row_bytes)
{
    return encode_tmap_2d(out128, CU_TENSOR_MAP_DATA_TYPE_UINT64, w, uint64_t(row_bytes / 8),
                          uint64_t(N), uint64_t(row_bytes), 18u, uint32_t(kTileRows),
                          CU_TENSOR_MAP_SWIZZLE_NONE);
}

} // namespace qmm
