// Host-only driver of the library's launch planners (no GPU needed): prints
// one JSON object per line for the shapes tests/test_host_plans.py asks
// about.  Linked against the library's object files; it calls only host
// functions that make no CUDA runtime call.
//
// Usage: host_plans <sm_count>
#include <cstdio>
#include <cstdlib>

#include "../quantized_gguf_dequant_gb300/csrc/qmm_internal.h"

int main(int argc, char **argv)
{
    const int sms = argc > 1 ? atoi(argv[1]) : 152;
    const long long Ns[] = {1, 16, 300, 512, 1024, 4096, 14336, 28672};
    const long long Ks[] = {256, 1024, 2048, 4096, 8192, 14336};
    for (long long N : Ns)
        for (long long K : Ks)
            for (int M = 1; M <= 16; ++M) {
                const qmm::TcbPlan p = qmm::plan_tcb(N, K, M, sms);
                printf("{\"kind\": \"tcb\", \"N\": %lld, \"K\": %lld, \"M\": %d, \"nt\": %d, "
                       "\"S\": %d, \"R\": %d, \"kc\": %d, \"smem\": %zu, \"ws_floats\": %zu, "
                       "\"tickets\": %zu}\n",
                       N, K, M, p.nt, p.S, p.R, p.kc, p.smem, p.ws_floats, p.tickets);
            }
    for (int tok : {128, 256})
        for (long long K : {1024LL, 4096LL, 14336LL})
            for (int tiles = 1; tiles <= 4 * sms + 7; ++tiles) {
                const qmm::GemmSplit g = qmm::gemm_q4k_split(tiles, tok, K, sms);
                printf("{\"kind\": \"gemm_split\", \"tiles\": %d, \"tok\": %d, \"K\": %lld, "
                       "\"full\": %d, \"ksplit\": %d}\n",
                       tiles, tok, K, g.full, g.ksplit);
            }
    for (long long M : {1LL, 100LL, 512LL, 2048LL})
        for (long long N : {1LL, 1024LL, 4096LL, 14336LL})
            for (int tok : {128, 256})
                printf("{\"kind\": \"gemm_tiles\", \"M\": %lld, \"N\": %lld, \"tok\": %d, "
                       "\"tiles\": %d, \"smem\": %zu}\n",
                       M, N, tok, qmm::gemm_q4k_tiles(M, N, tok), qmm::gemm_q4k_smem(tok, QMM_Q4_K));
    for (long long K : Ks)
        for (int M = 1; M <= 4; ++M)
            printf("{\"kind\": \"tc_smem\", \"K\": %lld, \"M\": %d, \"smem_16x2\": %zu, "
                   "\"smem_16x3\": %zu}\n",
                   K, M, qmm::gemv_tc_smem(K, M, 2, 16), qmm::gemv_tc_smem(K, M, 3, 16));
    for (int fmt : {int(QMM_Q4_K), int(QMM_Q8_0)})
        for (long long N : Ns)
            for (long long K : Ks) {
                const qmm::GemvPlan p = qmm::plan_gemv(fmt, N, K, sms, 0);
                printf("{\"kind\": \"gemv\", \"fmt\": %d, \"N\": %lld, \"K\": %lld, "
                       "\"kchunks\": %d, \"ksplit\": %d, \"rg\": %d, \"rpg\": %d, "
                       "\"stage_rows\": %d, \"stages\": %d, \"threads\": %d, "
                       "\"row_slices\": %d, \"slice_bytes\": %lld, \"smem\": %zu}\n",
                       fmt, N, K, p.kchunks, p.ksplit, p.rg, p.rpg, p.stage_rows, p.stages,
                       p.threads, p.row_slices, (long long)p.slice_bytes, p.smem);
            }
    // the no-allocation entry point's shapes: split-K scratch against the
    // static array
    const long long na[][2] = {{37, 2048}, {3000, 4096}, {5, 14336}, {16384, 1LL << 20}};
    for (int fmt : {int(QMM_Q4_K), int(QMM_Q8_0)})
        for (const auto &nk : na) {
            const qmm::GemvPlan p = qmm::plan_gemv(fmt, nk[0], nk[1], sms, 0);
            printf("{\"kind\": \"noalloc\", \"fmt\": %d, \"N\": %lld, \"K\": %lld, "
                   "\"ksplit\": %d, \"row_slices\": %d, \"need_floats\": %zu, "
                   "\"have_floats\": %zu, \"have_tickets\": %zu, \"fits\": %d}\n",
                   fmt, nk[0], nk[1], p.ksplit, p.row_slices,
                   qmm::gemv_workspace_floats(p, nk[0]), qmm::kNoallocPartialFloats,
                   qmm::kNoallocTickets, int(qmm::noalloc_fits(p, nk[0])));
        }
    // one-row decode kernel: tile counts of single matrices and groups,
    // every K-slice count (0 = the default choice)
    const long long Ts[] = {1, 2, 3, 16, 19, 64, 250, 256, 384, 1792, 8192, 20000};
    const long long NBs[] = {1, 2, 3, 4, 6, 7, 8, 12, 14, 16, 17, 28, 32, 56, 64};
    for (long long T : Ts)
        for (long long NB : NBs)
            for (int S : {0, 1, 2, 4, 7, 8, 16})
                for (int maxw : {8, 16}) {
                if (S > 0 && NB % S != 0)
                    continue;
                const qmm::M1Plan p = qmm::plan_m1(T, NB, sms, S, maxw);
                printf("{\"kind\": \"m1\", \"maxw\": %d, \"T\": %lld, \"NB\": %lld, \"force\": %d, "
                       "\"S\": %d, \"KS\": %d, \"WS\": %d, \"NP\": %d, \"TS\": %d, \"W\": %d, \"G1\": %d, "
                       "\"n_items\": %d, \"F\": %d, \"cap\": %d, \"nslot\": %d, "
                       "\"slot_bytes\": %d, \"smem\": %zu, \"smem_check\": %zu, "
                       "\"ws_floats\": %zu, \"tickets\": %zu}\n",
                       maxw, T, NB, S, p.S, p.KS, p.WS, p.NP, p.TS, p.W, p.G1, p.n_items, p.F, p.cap, p.nslot,
                       p.slot_bytes, p.smem, p.nslot ? qmm::m1_smem(p.KS, p.WS, p.TS, p.cap, p.nslot) : 0,
                       p.ws_floats, p.tickets);
            }
    return 0;
}
