// gemv_batched.cu -- Q4_K decode GEMV for a batch of activation rows
// (continuous batching: every row of X shares one read of the weights), on
// the tensor cores with the operand construction of gemv_tc.cu.
//
// The operation: "Frink Inference: the Rust alternative to llama.cpp",
// section "A serving stack with the full sampling surface" -- continuous
// batching runs the requests of one step through the weights together; with
// the dequantisation fused into the dot product ("Building a Rust Inference
// Engine That Matches Llama.cpp", "Where the wins came from").
//
//   Y[m][n] = sum_k w[n][k] * X[m][k],   m < M <= 16
//
// Up to 4*NT rows go through one pass: the A fragments of each k-step (the
// expensive part, built from the nibbles) feed NT mma.sync instructions, one
// per group of four rows.  The activations of all rows are re-laid out as B
// fragments in shared memory; since 16 rows of a long K do not fit, the grid
// is two-dimensional: CTA (r, s) owns row tiles [r*T/R, (r+1)*T/R) and
// super-blocks [s*NB/S, (s+1)*NB/S), so it prepares only its slice of X.
// With S > 1 the CTAs write partial sums per slice, added in slice order (so
// results are bitwise repeatable): for few partials per output (M*S <= 16)
// by the last CTA of each row group to finish (a ticket per row group), in
// the same launch; otherwise by a reduction kernel spread over the GPU.
#include <cstring>

#include <cuda.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "tc_common.cuh"

namespace qmm {

namespace {

using namespace tc;

struct TcbParams {
    CUtensorMap tmap;   // rows as 2-D uint64, box 18 x 16 (one unit)
    const float *x;     // [M][ldx]
    float *y;           // [M][ldy]
    float *ws;          // [S][M][N] partial sums (S > 1)
    unsigned *tickets;  // [R] arrivals per row group (in-kernel reduction; zero between launches)
    unsigned *status;
    int64_t ldx, ldy;
    int N, M, NB;
    int T;              // row tiles
    int R, S;           // row groups x K slices = grid
    int nslot;
};

// SB: one activation row (NT == 1, M == 1) with the per-sub-block operand
// form of tc_common.cuh (unit_dot_sb): unscaled subnormal nibbles, the
// sub-block scales applied once per sub-block.
template <int NT, bool SB>
__global__ void __launch_bounds__(256, 1) gemv_tcb_kernel(const __grid_constant__ TcbParams P)
{
    constexpr int NCOL = 8 * NT, MP = 4 * NT;
    extern __shared__ __align__(128) uint8_t smem[];
    const int nw = int(blockDim.x) >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int NS = P.nslot;
    const int r = blockIdx.x / P.S, s = blockIdx.x - r * P.S;
    const int t0 = int(int64_t(r) * P.T / P.R), t1 = int(int64_t(r + 1) * P.T / P.R);
    const int sb0 = int(int64_t(s) * P.NB / P.S), sb1 = int(int64_t(s + 1) * P.NB / P.S);
    const int KC = sb1 - sb0;

    uint8_t *ring = smem + size_t(warp) * NS * kTileBytes;
    uint8_t *acts = smem + size_t(nw) * NS * kTileBytes;
    uint2 *Bs = reinterpret_cast<uint2 *>(acts);                                   // [KC][16][NCOL][4]
    uint32_t *Bm = reinterpret_cast<uint32_t *>(Bs + size_t(KC) * 16 * NCOL * 4);   // [KC][NCOL][4]
    // SB: Bx [KC][16][4][2], the zero block Zx [16][8] and Xs [KC][8]
    uint2 *Bx = reinterpret_cast<uint2 *>(acts);
    uint2 *Zx = Bx + size_t(KC) * 128;
    float *Xs = reinterpret_cast<float *>(Zx + 128);
    float *inv = SB ? Xs + size_t(KC) * 8 : reinterpret_cast<float *>(Bm + size_t(KC) * NCOL * 4);  // [KC][MP]
    float *part = inv + size_t(KC) * MP;                                          // [nw][2][MP][16]
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(part + size_t(nw) * 2 * MP * kTileRows) + 7) & ~uintptr_t(7));
    uint64_t *bar = bars + warp * NS;
    __shared__ int wbeg[9];
    __shared__ unsigned s_last;

    const int cn = (t1 - t0) * KC;  // units of this CTA, ordered (tile, super-block)
    const int u0 = int(int64_t(warp) * cn / nw), u1 = int(int64_t(warp + 1) * cn / nw);
    const int nu = u1 - u0;
    if (lane == 0) {
        wbeg[warp] = u0;
        if (warp == nw - 1)
            wbeg[nw] = cn;
        for (int i = 0; i < NS; ++i)
            mbar_init(&bar[i], 1);
        fence_barrier_init();
    }
    __syncwarp();

    int i_tile = t0 + u0 / KC, i_sb = u0 % KC, slot_i = 0;
    auto issue = [&]() {
        mbar_arrive_expect_tx(&bar[slot_i], kTileBytes);
        tma_load_2d(ring + size_t(slot_i) * kTileBytes, &P.tmap, (sb0 + i_sb) * 18, i_tile * kTileRows,
                    &bar[slot_i], 0ull);
        if (++i_sb == KC) {
            i_sb = 0;
            ++i_tile;
        }
        if (++slot_i == NS)
            slot_i = 0;
    };
    int issued = nu < NS ? nu : NS;
    if (lane == 0)
        for (int j = 0; j < issued; ++j)
            issue();  // weights are constant: stream them before waiting on earlier kernels

    pdl_wait();

    // ---- this CTA's slice of every activation row -> B fragments (rows
    // beyond M are zeros, so every column is finite)
    {
        // Items (super-block, row) in rounds of eight per warp, their loads
        // in flight together.
        const int cc = lane >> 3, tt = lane & 7;
        const int items = KC * MP;
        for (int base = warp; base < items; base += 8 * nw) {
            float4 v[8], w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int item = base + i * nw;
                v[i] = w[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                const int sbl = item % KC, m = item / KC;
                if (item < items && m < P.M) {
                    const float *xr =
                        P.x + int64_t(m) * P.ldx + int64_t(sb0 + sbl) * 256 + 64 * cc + 4 * tt;
                    v[i] = __ldg(reinterpret_cast<const float4 *>(xr));
                    w[i] = __ldg(reinterpret_cast<const float4 *>(xr + 32));
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int item = base + i * nw;
                // One group of four: rows beyond M are not laid out (their
                // columns repeat real ones below); more groups: zeros.
                if constexpr (SB) {
                    if (item < KC)
                        prep_super_block_sb(item, v[i], w[i], lane, Bx, Xs, inv);
                } else if (item < items && (NT > 1 || item / KC < P.M)) {
                    prep_super_block<NCOL>(item % KC, item / KC, MP, v[i], w[i], lane, Bs, Bm, inv);
                }
            }
        }
        if constexpr (SB)
            for (int i = threadIdx.x; i < 128; i += blockDim.x)
                Zx[i] = make_uint2(0u, 0u);
    }
    __syncthreads();

    uint32_t selA, selB;
    bool hi4;
    chunk_selectors(c, selA, selB, hi4);
    const uint8_t *rowA = ring + g * 144;
    float *mypart = part + size_t(warp) * 2 * MP * kTileRows;
    // B column of this lane: with one group of four and M < 4, columns
    // beyond 2M repeat real ones (finite; their outputs are never stored).
    const bool bact = (g >> 1) == c;  // SB: this lane reads a B entry (else the zero block)
    const int boff = 2 * c + (g & 1);
    const int col = NT == 1 ? g % (2 * P.M) : g;
    const int cinv = NT == 1 && c >= P.M ? 0 : c;
    // One output (row tile t, rows rr and rr+8, activation row m): to Y, or to
    // this slice's partial sums.
    auto emit = [&](int t, int rr, int m, float v0, float v1) {
        if (m >= P.M)
            return;
        const int row = t * kTileRows + rr;
        float *dst = P.S > 1 ? P.ws + (int64_t(s) * P.M + m) * P.N : P.y + int64_t(m) * P.ldy;
        if (row < P.N)
            dst[row] = v0;
        if (row + 8 < P.N)
            dst[row + 8] = v1;
    };

    float tot0[NT], tot1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        tot0[nt] = tot1[nt] = 0.f;
    int q_tile = t0 + u0 / KC, q_sb = u0 % KC;
    int slot = 0;
    unsigned parity = 0;
    int jfail = -1;
    for (int j = 0; j < nu; ++j) {
        if (!mbar_wait_bounded(&bar[slot], parity)) {
            jfail = j;
            break;
        }
        if constexpr (SB) {
            const uint2 *bx = bact ? Bx + (size_t(q_sb) * 128 + boff) : Zx;
            const float2 xab = *reinterpret_cast<const float2 *>(Xs + q_sb * 8 + 2 * c);
            unit_dot_sb(rowA + slot * kTileBytes, c, selA, selB, hi4, bx, xab, inv[q_sb], tot0[0],
                        tot1[0]);
        } else {
            unit_dot_nt<NT>(rowA + slot * kTileBytes, c, selA, selB, hi4,
                            Bs + (size_t(q_sb) * 16 * NCOL + col) * 4 + c,
                            Bm + (size_t(q_sb) * NCOL + col) * 4 + c, inv + q_sb * MP + cinv, tot0,
                            tot1);
        }
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
        const int ju = u0 + j;
        if (q_sb == KC - 1 || j == nu - 1) {
            if constexpr (SB) {
                // The four lanes of a row pair hold two sub-blocks each.
                tot0[0] += __shfl_xor_sync(0xffffffffu, tot0[0], 1);
                tot1[0] += __shfl_xor_sync(0xffffffffu, tot1[0], 1);
                tot0[0] += __shfl_xor_sync(0xffffffffu, tot0[0], 2);
                tot1[0] += __shfl_xor_sync(0xffffffffu, tot1[0], 2);
            }
            const int first = (ju / KC) * KC, last = first + KC - 1;
            if (u0 <= first && u1 - 1 >= last) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    emit(q_tile, g, 4 * nt + c, tot0[nt], tot1[nt]);
            } else {
                const int k = (u0 >= first) ? 0 : 1;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mypart[(k * MP + 4 * nt + c) * kTileRows + g] = tot0[nt];
                    mypart[(k * MP + 4 * nt + c) * kTileRows + g + 8] = tot1[nt];
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                tot0[nt] = tot1[nt] = 0.f;
        }
        if (++q_sb == KC) {
            q_sb = 0;
            ++q_tile;
        }
    }
    if (jfail >= 0 && lane == 0) {
        atomicOr(P.status, kStatusTimeoutBit);
        for (int j = jfail; j < issued; ++j)
            mbar_wait_bounded(&bar[j % NS], unsigned(j / NS) & 1u, 100000000ll);
    }
    pdl_launch_dependents();
    __syncthreads();

    // ---- tiles split between warps: add the shares in warp order
    {
        const int cm = lane >> 3, cr = lane & 7;
        for (int tr = warp; tr < t1 - t0; tr += nw) {
            const int first = tr * KC, last = first + KC - 1;
            int wf = 0, wl = 0;
            for (int w = 0; w < nw; ++w) {
                if (wbeg[w] <= first)
                    wf = w;
                if (wbeg[w] <= last)
                    wl = w;
            }
            if (wf == wl)
                continue;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float s0 = 0.f, s1 = 0.f;
                for (int w = wf; w <= wl; ++w) {
                    const int b0 = wbeg[w], b1 = wbeg[w + 1];
                    if (b1 == b0)
                        continue;
                    const int kw = (b0 >= first) ? 0 : 1;
                    const float *pw = part + (size_t(w) * 2 + kw) * MP * kTileRows +
                                      (4 * nt + cm) * kTileRows;
                    s0 += pw[cr];
                    s1 += pw[cr + 8];
                }
                emit(t0 + tr, cr, 4 * nt + cm, s0, s1);
            }
        }
    }
    if (P.S == 1 || !P.tickets)
        return;

    // ---- K slices: the row group's last CTA to arrive adds the S partial
    // sums of its rows in slice order and resets the ticket.
    __threadfence();  // this thread's partial sums, device-wide, before the ticket
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atomicAdd(&P.tickets[r], 1u) == unsigned(P.S - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    const int row0 = t0 * kTileRows, row1 = min(t1 * kTileRows, P.N), nr = row1 - row0;
    const int64_t slice = int64_t(P.M) * P.N;
    for (int i = threadIdx.x; i < P.M * nr; i += blockDim.x) {
        const int m = i / nr, row = row0 + (i - m * nr);
        const float *src = P.ws + int64_t(m) * P.N + row;
        float acc = __ldcg(src);
        for (int k = 1; k < P.S; ++k)
            acc += __ldcg(src + k * slice);
        P.y[int64_t(m) * P.ldy + row] = acc;
    }
    if (threadIdx.x == 0)
        P.tickets[r] = 0u;
}

// y[m][n] = ws[0][m][n] + ... + ws[S-1][m][n], in slice order.
__global__ void tcb_reduce_kernel(const float *__restrict__ ws, int S, int M, int N,
                                  float *__restrict__ y, int64_t ldy)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t n_all = int64_t(M) * N, stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_all; i += stride) {
        float acc = __ldcs(ws + i);
        for (int k = 1; k < S; ++k)
            acc += __ldcs(ws + int64_t(k) * n_all + i);
        const int64_t m = i / N;
        y[m * ldy + (i - m * N)] = acc;
    }
}

using TcbKernel = void (*)(TcbParams);

TcbKernel pick_tcb(int nt, bool sb)
{
    switch (nt) {
    case 1: return sb ? gemv_tcb_kernel<1, true> : gemv_tcb_kernel<1, false>;
    case 2: return gemv_tcb_kernel<2, false>;
    case 3: return gemv_tcb_kernel<3, false>;
    default: return gemv_tcb_kernel<4, false>;
    }
}

constexpr int kTcbWarps = 8;
// Largest M*S whose slices one CTA per row group adds at the end of the main
// launch (measured: M = 1 with four slices gains; M = 8 and 16 with 4-14
// slices lose against the separate reduction).
constexpr int kTcbInKernelPartials = 16;
constexpr int kTcbMaxSlots = 8;

// Ring slots per warp: 2 (a sweep of 2, 3, 4 and 6 on the decode step and
// the batched sweep put 2-3 first); QMM_TCB_NSLOT overrides, 2..8.
int tcb_slots()
{
    const char *e = getenv("QMM_TCB_NSLOT");
    if (e && atoi(e) >= 2 && atoi(e) <= kTcbMaxSlots)
        return atoi(e);
    return 2;
}

size_t tcb_smem(int nt, int kc, bool sb)
{
    const size_t ncol = 8 * nt, mp = 4 * nt;
    const int ns = tcb_slots();
    const size_t acts = sb ? size_t(kc) * 128 * 8 + 128 * 8 + size_t(kc) * 8 * 4
                           : size_t(kc) * 16 * ncol * 4 * 8 + size_t(kc) * ncol * 4 * 4;
    return size_t(kTcbWarps) * ns * kTileBytes + acts + size_t(kc) * mp * 4 +
           size_t(kTcbWarps) * 2 * mp * kTileRows * 4 + 8 + size_t(kTcbWarps) * ns * 8;
}

} // namespace

// Grid plan: rows per pass up to 16 (NT = ceil(M/4) groups of four); K split
// into S slices of at most 16/NT super-blocks, so a CTA lays out at most 64
// (super-block, row) activation items -- one round of eight per warp -- and
// into more slices when there are too few row tiles to cover the SMs; about
// one CTA per SM: R = SMs / S row groups (at most one per row tile).  The
// work per CTA does not depend on S; the partial sums (S x M x N floats) do.
// QMM_TCB_S forces S (at least the number that fits).
TcbPlan plan_tcb(int64_t N, int64_t K, int M, int sm_count)
{
    TcbPlan p;
    p.nt = (M + 3) / 4;
    const int NB = int(K / 256);
    const int T = int((N + kTileRows - 1) / kTileRows);
    int kcmax = 0;
    const bool sb = M == 1;
    while (kcmax < NB && tcb_smem(p.nt, kcmax + 1, sb) <= size_t(227 * 1024))
        ++kcmax;
    if (kcmax == 0)
        return p;
    // One round of eight activation items per warp: KC * 4 * NT <= 64.
    int kc = 16 / p.nt;
    if (kc > kcmax)
        kc = kcmax;
    if (kc > NB)
        kc = NB;
    p.S = (NB + kc - 1) / kc;
    if (const char *e = getenv("QMM_TCB_S")) {
        const int f = atoi(e);
        if (f >= (NB + kcmax - 1) / kcmax && f <= NB)
            p.S = f;
    }
    // Few row tiles: slice K further so that the grid still covers the SMs.
    if (!getenv("QMM_TCB_S") && p.S * T < sm_count) {
        const int want = sm_count / T;
        if (want > p.S)
            p.S = want < NB ? want : NB;
    }
    p.R = sm_count / p.S;
    if (p.R < 1)
        p.R = 1;
    if (p.R > T)
        p.R = T;
    p.kc = (NB + p.S - 1) / p.S;
    p.smem = tcb_smem(p.nt, p.kc, sb);
    p.ws_floats = p.S > 1 ? size_t(p.S) * size_t(M) * size_t(N) : 0;
    p.tickets = (p.S > 1 && M * p.S <= kTcbInKernelPartials) ? size_t(p.R) : 0;
    return p;
}

cudaError_t launch_gemv_tcb(const TcbArgs &a, const TcbPlan &p, cudaStream_t s)
{
    TcbParams P;
    memset(&P, 0, sizeof(P));
    P.tmap = *reinterpret_cast<const CUtensorMap *>(a.tmap);
    P.x = a.x;
    P.y = a.y;
    P.ws = a.ws;
    P.tickets = p.tickets ? a.tickets : nullptr;
    P.status = a.status;
    P.ldx = a.ldx;
    P.ldy = a.ldy;
    P.N = int(a.N);
    P.M = a.M;
    P.NB = int(a.K / 256);
    P.T = int((a.N + kTileRows - 1) / kTileRows);
    P.R = p.R;
    P.S = p.S;
    P.nslot = tcb_slots();
    TcbKernel kern = pick_tcb(p.nt, a.M == 1);
    cudaError_t e = func_smem(reinterpret_cast<const void *>(kern), p.smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.R * p.S));
    cfg.blockDim = dim3(unsigned(kTcbWarps * 32));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    e = counted(cudaLaunchKernelEx(&cfg, kern, P));
    if (e != cudaSuccess || p.S == 1 || p.tickets)
        return e;
    const int64_t n = int64_t(a.M) * a.N;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = int64_t(p.R) * p.S * 8;
    if (blocks > cap)
        blocks = cap;
    cudaLaunchConfig_t rc = cfg;
    rc.gridDim = dim3(unsigned(blocks));
    rc.blockDim = dim3(256);
    rc.dynamicSmemBytes = 0;
    return counted(cudaLaunchKernelEx(&rc, tcb_reduce_kernel, static_cast<const float *>(a.ws), p.S,
                                      a.M, int(a.N), a.y, a.ldy));
}

} // namespace qmm
