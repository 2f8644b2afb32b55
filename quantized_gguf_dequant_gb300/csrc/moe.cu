// moe.cu -- mixture-of-experts layers on the Q4_K tensor-core GEMV.
//
// The operation: "Frink Inference: the Rust alternative to llama.cpp",
// sections "The goal, stated once" and "Architecture coverage: 100 models
// with evidence" -- mixture-of-experts checkpoints, whose feed-forward block
// sends each token through the top_k experts its router picked and sums their
// outputs with the router's weights.  Per token t and slot s with expert
// e = ids[t, s]:  g = Wg_e x_t, u = Wu_e x_t, h = silu(g) * u,
// y_t = sum_s r[t, s] * Wd_e h.  Llama 4 applies r to the expert's input
// instead ("Architecture coverage: 100 models with evidence": the expert
// weight applied to the input of the expert): g = Wg_e (r x_t),
// u = Wu_e (r x_t), y_t = sum_s Wd_e h -- the expert step scales each
// slot's activations by r as it loads them, the combine adds without r.
//
// Steps, one kernel each:
//  1. bucket   -- one CTA sorts the T*top_k slots by expert id (stable, so
//                 the order is fixed) and cuts every expert's slots into
//                 groups of at most kGroupTokens.  Ids outside
//                 [0, n_experts) are dropped and flagged in the status word.
//  2. expert   -- the tensor-core GEMV of gemv_tc.cu, with a group's tokens
//                 as the activation rows.  Work = (group, 16-row tile,
//                 super-block) units; every expert's rows are read from HBM
//                 by its first group, later groups of the same expert
//                 re-read them while they are still in L2.  Gate and up run
//                 in one launch (two matrices, one set of groups).
//  3. swiglu   -- h = silu(g) * u, elementwise.
//  4. combine  -- y_t = sum_s r[t, s] * y_(t,s), slot order, skipping
//                 dropped slots.
// No step uses atomics on data, so every result is bitwise repeatable.
#include <algorithm>
#include <cstring>

#include <cuda.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "tc_common.cuh"

namespace qmm {

namespace {

using namespace tc;

constexpr int kNcol = 8;  // B columns: kGroupTokens rows x (hi, lo)

// ------------------------------------------------------------------ bucket

// ids: [S] int32.  Writes, for E = n_experts:
//   slots[0 .. S')       valid slots sorted by (expert, slot)
//   groups[0 .. G)       int4 {expert, first index into slots, count, 0}
//   *n_groups            G
// and, when y0 != nullptr, zeroes row s of y0 ([S, ld0] floats, n0 of them)
// for every dropped slot s.
__global__ void __launch_bounds__(1024) moe_bucket_kernel(const int32_t *__restrict__ ids, int S,
                                                          int E, int4 *groups, int *slots,
                                                          int *n_groups, float *y0, int64_t n0,
                                                          int64_t ld0, unsigned *status)
{
    extern __shared__ int sm_bucket[];
    int *sid = sm_bucket;       // [S]
    int *cnt = sid + S;         // [E]
    int *off = cnt + E;         // [E] first index into slots
    int *goff = off + E;        // [E] first group
    __shared__ int bad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (threadIdx.x == 0)
        bad = 0;
    __syncthreads();
    pdl_wait();
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int e = ids[s];
        sid[s] = e;
        if (e < 0 || e >= E)
            bad = 1;
    }
    __syncthreads();
    pdl_launch_dependents();
    // Counts: warp w handles experts w, w+nw, ...
    for (int e = warp; e < E; e += nw) {
        int n = 0;
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            n += __popc(__ballot_sync(0xffffffffu, s < S && sid[s] == e));
        }
        if (lane == 0)
            cnt[e] = n;
    }
    __syncthreads();
    // Exclusive prefix sums of counts and group counts (warp 0; each lane
    // takes a contiguous run of experts).
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int a = 0, b = 0;
        for (int e = e0; e < e1; ++e) {
            a += cnt[e];
            b += (cnt[e] + kGroupTokens - 1) / kGroupTokens;
        }
        int ia = a, ib = b;  // inclusive scan over lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, ia, o);
            const int tb = __shfl_up_sync(0xffffffffu, ib, o);
            if (lane >= o) {
                ia += ta;
                ib += tb;
            }
        }
        int ra = ia - a, rb = ib - b;
        for (int e = e0; e < e1; ++e) {
            off[e] = ra;
            goff[e] = rb;
            ra += cnt[e];
            rb += (cnt[e] + kGroupTokens - 1) / kGroupTokens;
        }
        if (lane == 31)
            *n_groups = ib;
    }
    __syncthreads();
    // Slot lists (ascending slot order within an expert) and group records.
    for (int e = warp; e < E; e += nw) {
        int pos = off[e];
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            const bool hit = s < S && sid[s] == e;
            const unsigned mask = __ballot_sync(0xffffffffu, hit);
            if (hit)
                slots[pos + __popc(mask & ((1u << lane) - 1u))] = s;
            pos += __popc(mask);
        }
        const int ng = (cnt[e] + kGroupTokens - 1) / kGroupTokens;
        for (int j = lane; j < ng; j += 32)
            groups[goff[e] + j] =
                make_int4(e, off[e] + j * kGroupTokens, min(kGroupTokens, cnt[e] - j * kGroupTokens), 0);
    }
    if (bad) {
        if (threadIdx.x == 0)
            atomicOr(status, kStatusBadExpertBit);
        if (y0) {
            for (int s = warp; s < S; s += nw) {
                const int e = sid[s];
                if (e < 0 || e >= E)
                    for (int64_t n = lane; n < n0; n += 32)
                        y0[int64_t(s) * ld0 + n] = 0.f;
            }
        }
    }
}

// ------------------------------------------------------------------ expert GEMV

struct MoeParams {
    CUtensorMap tmap[2];       // the stacked expert matrices (n_experts * Ne rows)
    float *y[2];               // per-slot outputs [S][Ne] of each matrix
    const float *x;            // activations
    int64_t ldx;
    const int4 *groups;
    const int *slots;
    const int *n_groups;
    unsigned *status;
    int Ne;                    // rows per expert
    int tpm;                   // row tiles per expert and matrix, ceil(Ne / 16)
    int nmat;                  // 1 or 2
    int NB;                    // super-blocks per row
    int top_k;
    int x_per_slot;
    const float *xscale;       // per-slot input scale [S] (routing on the input), or null
    int nslot;
    // fuse = 1 (nmat = 2, gate and up): tiles are taken in (gate, up) pairs
    // of the same rows, staged in shared memory (room for maxpairs pairs per
    // CTA) and y[0] receives h = silu(gate) * up instead of either product.
    int fuse;
    int maxpairs;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// One CTA: an even share of the (group, tile) sequence; within it, one
// segment per group, each computed like the decode GEMV (warps split the
// segment's units; shared tiles are added in shared memory in warp order).
__global__ void __launch_bounds__(512, 1) moe_expert_kernel(const __grid_constant__ MoeParams P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int nw = int(blockDim.x) >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int NB = P.NB, NS = P.nslot;

    uint8_t *ring = smem + size_t(warp) * NS * kTileBytes;
    uint2 *Bs = reinterpret_cast<uint2 *>(smem + size_t(nw) * NS * kTileBytes);  // [NB][16][8][4]
    uint32_t *Bm = reinterpret_cast<uint32_t *>(Bs + size_t(NB) * 16 * kNcol * 4);  // [NB][8][4]
    float *inv = reinterpret_cast<float *>(Bm + size_t(NB) * kNcol * 4);            // [NB][4]
    float *part = inv + size_t(NB) * kGroupTokens;                                 // [nw][2][4][16]
    float *res = part + size_t(nw) * 2 * 4 * kTileRows;  // fused: [2*maxpairs][4][16] tile results
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(res + size_t(P.fuse ? 2 * P.maxpairs : 0) * 4 * kTileRows) + 7) &
        ~uintptr_t(7));
    uint64_t *bar = bars + warp * NS;
    __shared__ int wbeg[17];
    __shared__ int gslot[kGroupTokens];

    if (lane == 0) {
        for (int s = 0; s < NS; ++s)
            mbar_init(&bar[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    pdl_wait();  // the bucket tables, x and y belong to earlier kernels until here
    pdl_launch_dependents();

    const int tilesG = P.nmat * P.tpm;             // tiles per group
    const int64_t Ttot = int64_t(*P.n_groups) * tilesG;
    const int64_t G = gridDim.x;
    // Fused: CTAs take whole (gate, up) pairs, so the split is over pairs.
    const int64_t unit_tiles = P.fuse ? 2 : 1;
    const int64_t Tsplit = Ttot / unit_tiles;
    const int64_t t0 = (blockIdx.x * Tsplit / G) * unit_tiles,
                  t1 = ((blockIdx.x + 1) * Tsplit / G) * unit_tiles;
    // Local tile of a group -> (matrix, 16-row tile of the expert).
    auto tile_mat = [&](int lt, int &mat, int &rt) {
        if (P.fuse) {
            mat = lt & 1;
            rt = lt >> 1;
        } else {
            mat = lt >= P.tpm ? 1 : 0;
            rt = lt - mat * P.tpm;
        }
    };

    uint32_t selA, selB;
    bool hi4;
    chunk_selectors(c, selA, selB, hi4);
    const int col = g;     // B column of this lane's fragments
    const int mrow = c;    // group token whose two terms sit in this lane's accumulator columns
    const uint8_t *rowA = ring + g * 144;
    float *mypart = part + size_t(warp) * 2 * 4 * kTileRows;
    // Copies are numbered per warp across segments: copy n uses slot n % NS
    // and completes phase (n / NS) & 1 of that slot's barrier.
    int gbase = 0;  // copies of this warp before the current segment
    __shared__ int s_fail;
    if (threadIdx.x == 0)
        s_fail = 0;
    bool failed = false;

    for (int64_t ts = t0; ts < t1 && !failed;) {
        // ---- segment: tiles [ts, te) of group gi
        const int gi = int(ts / tilesG);
        const int64_t te = min(t1, int64_t(gi + 1) * tilesG);
        const int4 grp = P.groups[gi];  // {expert, first, count}
        const int lt0 = int(ts - int64_t(gi) * tilesG);
        const int cn = int(te - ts) * NB;  // units of the segment
        const int u0 = warp * cn / nw, u1 = (warp + 1) * cn / nw;
        const int nu = u1 - u0;
        if (lane == 0) {
            wbeg[warp] = u0;
            if (warp == nw - 1)
                wbeg[nw] = cn;
        }
        if (threadIdx.x < kGroupTokens)
            gslot[threadIdx.x] = threadIdx.x < grp.z ? P.slots[grp.y + threadIdx.x] : -1;

        // Unit u of the segment: local tile lt0 + u / NB, super-block u % NB.
        int i_tile = lt0 + u0 / NB, i_sb = u0 % NB;
        int slot_i = gbase % NS;
        auto issue = [&]() {
            int mat, lt;
            tile_mat(i_tile, mat, lt);
            mbar_arrive_expect_tx(&bar[slot_i], kTileBytes);
            tma_load_2d(ring + size_t(slot_i) * kTileBytes, &P.tmap[mat], i_sb * 18,
                        grp.x * P.Ne + lt * kTileRows, &bar[slot_i], 0ull);
            if (++i_sb == NB) {
                i_sb = 0;
                ++i_tile;
            }
            if (++slot_i == NS)
                slot_i = 0;
        };
        int issued = nu < NS ? nu : NS;
        if (lane == 0)
            for (int j = 0; j < issued; ++j)
                issue();

        __syncthreads();  // gslot visible; the previous segment's B no longer read

        // ---- activations of the group's tokens -> B fragments (zeros for
        // absent tokens, so every column is finite)
        {
            const int cc = lane >> 3, tt = lane & 7;
            for (int item = warp; item < NB * kGroupTokens; item += nw) {
                const int sb = item % NB, m = item / NB;
                const int s = gslot[m];
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f), w = v;
                if (s >= 0) {
                    const int64_t xrow = P.x_per_slot ? s : s / P.top_k;
                    const float *xr = P.x + xrow * P.ldx + int64_t(sb) * 256 + 64 * cc + 4 * tt;
                    v = __ldg(reinterpret_cast<const float4 *>(xr));
                    w = __ldg(reinterpret_cast<const float4 *>(xr + 32));
                    if (P.xscale) {  // the slot's routing weight on its input
                        const float r = __ldg(P.xscale + s);
                        v = make_float4(r * v.x, r * v.y, r * v.z, r * v.w);
                        w = make_float4(r * w.x, r * w.y, r * w.z, r * w.w);
                    }
                }
                prep_super_block<kNcol>(sb, m, kGroupTokens, v, w, lane, Bs, Bm, inv);
            }
        }
        __syncthreads();

        // ---- main loop over this warp's units
        float tot0 = 0.f, tot1 = 0.f;
        int q_tile = lt0 + u0 / NB, q_sb = u0 % NB;
        int slot = gbase % NS;
        unsigned parity = unsigned(gbase / NS) & 1u;
        int jfail = -1;
        for (int j = 0; j < nu; ++j) {
            if (!mbar_wait_bounded(&bar[slot], parity)) {
                jfail = j;
                break;
            }
            unit_dot<kNcol>(rowA + slot * kTileBytes, c, selA, selB, hi4,
                            Bs + (size_t(q_sb) * 16 * kNcol + col) * 4 + c,
                            Bm[(size_t(q_sb) * kNcol + col) * 4 + c], inv[q_sb * kGroupTokens + mrow],
                            tot0, tot1);
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
            const int ju = u0 + j;  // unit index within the segment
            if (q_sb == NB - 1 || j == nu - 1) {
                const int first = (ju / NB) * NB, last = first + NB - 1;
                if (u0 <= first && u1 - 1 >= last) {
                    const int s = gslot[mrow];
                    if (P.fuse) {
                        float *rr = res + (size_t(q_tile - lt0) * 4 + mrow) * kTileRows;
                        rr[g] = tot0;
                        rr[g + 8] = tot1;
                    } else if (s >= 0) {
                        int mat, rt;
                        tile_mat(q_tile, mat, rt);
                        const int r = rt * kTileRows + g;
                        float *yr = P.y[mat] + int64_t(s) * P.Ne;
                        if (r < P.Ne)
                            yr[r] = tot0;
                        if (r + 8 < P.Ne)
                            yr[r + 8] = tot1;
                    }
                } else {
                    const int k = (u0 >= first) ? 0 : 1;
                    mypart[(k * 4 + mrow) * kTileRows + g] = tot0;
                    mypart[(k * 4 + mrow) * kTileRows + g + 8] = tot1;
                }
                tot0 = tot1 = 0.f;
            }
            if (++q_sb == NB) {
                q_sb = 0;
                ++q_tile;
            }
        }
        if (jfail >= 0 && lane == 0) {
            atomicOr(P.status, kStatusTimeoutBit);
            s_fail = 1;
            // Let this warp's copies in flight land before shared memory is released.
            for (int j = jfail; j < issued; ++j)
                mbar_wait_bounded(&bar[(gbase + j) % NS], unsigned((gbase + j) / NS) & 1u,
                                  100000000ll);
        }
        __syncthreads();
        failed = s_fail != 0;  // the same for every thread of the CTA

        // ---- tiles no single warp covered: add the warps' shares in warp order
        const int cm = lane >> 3, cr = lane & 7;
        const int ntile = int(te - ts);
        for (int tr = warp; tr < ntile && !failed; tr += nw) {
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
                continue;
            float s0 = 0.f, s1 = 0.f;
            for (int w = wf; w <= wl; ++w) {
                const int b0 = wbeg[w], b1 = wbeg[w + 1];
                if (b1 == b0)
                    continue;
                const int kw = (b0 >= first) ? 0 : 1;
                const float *pw = part + (size_t(w) * 2 + kw) * 4 * kTileRows + cm * kTileRows;
                s0 += pw[cr];
                s1 += pw[cr + 8];
            }
            const int s = gslot[cm];
            if (P.fuse) {
                float *rr = res + (size_t(tr) * 4 + cm) * kTileRows;
                rr[cr] = s0;
                rr[cr + 8] = s1;
            } else if (s >= 0) {
                int mat, rt;
                tile_mat(lt0 + tr, mat, rt);
                const int r = rt * kTileRows + cr;
                float *yr = P.y[mat] + int64_t(s) * P.Ne;
                if (r < P.Ne)
                    yr[r] = s0;
                if (r + 8 < P.Ne)
                    yr[r + 8] = s1;
            }
        }
        if (P.fuse && !failed) {
            // ---- h = silu(gate) * up for every (pair, token, row) of the segment
            __syncthreads();
            const int npair = ntile / 2;
            for (int i = threadIdx.x; i < npair * 4 * kTileRows; i += blockDim.x) {
                const int pl = i / (4 * kTileRows), m = (i / kTileRows) & 3, rr = i % kTileRows;
                const int s = gslot[m];
                const int r = ((lt0 >> 1) + pl) * kTileRows + rr;
                if (s < 0 || r >= P.Ne)
                    continue;
                const float gv = res[(size_t(2 * pl) * 4 + m) * kTileRows + rr];
                const float uv = res[(size_t(2 * pl + 1) * 4 + m) * kTileRows + rr];
                P.y[0][int64_t(s) * P.Ne + r] = silu(gv) * uv;
            }
        }
        gbase += nu;
        __syncthreads();  // part[], wbeg[] and gslot[] are reused by the next segment
        ts = te;
    }
}

// ------------------------------------------------------------------ elementwise

__global__ void swiglu_kernel(const float *__restrict__ g, const float *__restrict__ u,
                              float *__restrict__ h, int64_t n)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        h[i] = silu(g[i]) * u[i];
}

// y[t][n] = sum_s r[t][s] * ys[t*top_k + s][n], s ascending; dropped slots
// (ids outside [0, E)) contribute nothing.  r == nullptr: the plain sum (the
// routing weight was applied to the experts' inputs).
__global__ void moe_combine_kernel(const float *__restrict__ ys, const float *__restrict__ r,
                                   const int32_t *__restrict__ ids, int E, int T, int top_k,
                                   int64_t Ne, float *__restrict__ y)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t total = int64_t(T) * Ne;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / Ne, n = i - t * Ne;
        float acc = 0.f;
        for (int s = 0; s < top_k; ++s) {
            const int64_t slot = t * top_k + s;
            const int e = ids[slot];
            if (e >= 0 && e < E)
                acc = r ? fmaf(r[slot], ys[slot * Ne + n], acc) : acc + ys[slot * Ne + n];
        }
        y[i] = acc;
    }
}

template <typename Kernel, typename... Args>
cudaError_t launch_ex(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return counted(cudaLaunchKernelEx(&cfg, k, args...));
}

} // namespace

size_t moe_bucket_smem(int S, int E) { return size_t(S + 3 * E) * sizeof(int); }

cudaError_t launch_moe_bucket(const int32_t *ids, int S, int E, const MoeIndex &ix, float *y0,
                              int64_t n0, int64_t ld0, unsigned *status, cudaStream_t s)
{
    const size_t smem = moe_bucket_smem(S, E);
    cudaError_t e = func_smem(reinterpret_cast<const void *>(moe_bucket_kernel), smem);
    if (e != cudaSuccess)
        return e;
    return launch_ex(moe_bucket_kernel, dim3(1), dim3(1024), smem, s, ids, S, E, ix.groups,
                     ix.slots, ix.n_groups, y0, n0, ld0, status);
}

void moe_expert_shape(int64_t K, int &nw, int &nslot)
{
    nw = 16;
    nslot = 2;  // measured on the OLMoE layer: 16 x 2 ahead of 16 x 3/4, 12 x 2, 8 x 4
    const char *ew = getenv("QMM_MOE_WARPS"), *es = getenv("QMM_MOE_NSLOT");
    if (ew && atoi(ew) > 0)
        nw = atoi(ew);
    if (es && atoi(es) > 0)
        nslot = atoi(es);
    if (!(ew || es) && moe_expert_smem(K, nw, nslot, 0) > size_t(227 * 1024)) {
        nw = 8;
        nslot = 4;
    }
}

size_t moe_expert_smem(int64_t K, int nw, int nslot, int maxpairs)
{
    const size_t NB = size_t(K / 256);
    size_t b = size_t(nw) * nslot * kTileBytes;
    b += NB * 16 * kNcol * 4 * sizeof(uint2);
    b += NB * kNcol * 4 * sizeof(uint32_t);
    b += NB * kGroupTokens * sizeof(float);
    b += size_t(nw) * 2 * 4 * kTileRows * sizeof(float);
    b += size_t(2 * maxpairs) * 4 * kTileRows * sizeof(float);
    b = (b + 7) & ~size_t(7);
    b += size_t(nw) * nslot * sizeof(uint64_t);
    return b;
}

cudaError_t launch_moe_expert(const MoeExpertArgs &a, int sm_count, cudaStream_t s)
{
    MoeParams P;
    memset(&P, 0, sizeof(P));
    for (int i = 0; i < a.nmat; ++i) {
        memcpy(&P.tmap[i], a.tmap[i], sizeof(CUtensorMap));
        P.y[i] = a.y[i];
    }
    P.x = a.x;
    P.ldx = a.ldx;
    P.groups = a.ix.groups;
    P.slots = a.ix.slots;
    P.n_groups = a.ix.n_groups;
    P.status = a.status;
    P.Ne = int(a.Ne);
    P.tpm = int((a.Ne + kTileRows - 1) / kTileRows);
    P.nmat = a.nmat;
    P.NB = int(a.K / 256);
    P.top_k = a.top_k;
    P.x_per_slot = a.x_per_slot;
    P.xscale = a.xscale;
    P.fuse = a.fuse_swiglu;
    P.maxpairs = a.fuse_swiglu ? a.maxpairs : 0;
    int nw, nslot;
    moe_expert_shape(a.K, nw, nslot);
    P.nslot = nslot;
    const size_t smem = moe_expert_smem(a.K, nw, nslot, P.maxpairs);
    cudaError_t e = func_smem(reinterpret_cast<const void *>(moe_expert_kernel), smem);
    if (e != cudaSuccess)
        return e;
    // The number of groups is known only on the device: one CTA per SM, each
    // takes an even share of whatever the bucketing produced.
    return launch_ex(moe_expert_kernel, dim3(sm_count), dim3(32 * nw), smem, s, P);
}

cudaError_t launch_swiglu(const float *g, const float *u, float *h, int64_t n, int sm_count,
                          cudaStream_t s)
{
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, int64_t(sm_count) * 8);
    return launch_ex(swiglu_kernel, dim3(unsigned(std::max<int64_t>(blocks, 1))), dim3(256), 0,
                     s, g, u, h, n);
}

cudaError_t launch_moe_combine(const float *ys, const float *r, const int32_t *ids, int E, int T,
                               int top_k, int64_t Ne, float *y, int sm_count, cudaStream_t s)
{
    const int64_t total = int64_t(T) * Ne;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, int64_t(sm_count) * 8);
    return launch_ex(moe_combine_kernel, dim3(unsigned(std::max<int64_t>(blocks, 1))), dim3(256),
                     0, s, ys, r, ids, E, T, top_k, Ne, y);
}

} // namespace qmm
