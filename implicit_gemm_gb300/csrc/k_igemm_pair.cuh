// The x-taps-on-columns tile of igemm_wgrad_kernel on a pair of SMs
// (tcgen05 .cta_group::2).
//
// With the x taps on the columns a split's D[(y, c), (x, k)] is two M-tiles of
// 128 rows (atoms y = 0, 1 and y = 2, 3 or padding) by N = 64*X columns.  Run
// as two separate CTAs (igemm_wgrad_kernel), each SM stages the whole dY patch
// and reads A (4 KB) and all of B (32*N bytes) from its shared memory for
// every 16-pixel K-step: with 3x3 filters ~234 KB per 256-pixel K-tile through
// shared memory against ~1.5k cycles of tensor work, so the main loop runs at
// the shared-memory rate rather than the tensor rate.
//
// Here the two CTAs of a split form a cluster and share M = 256 MMAs issued by
// rank 0: rank r holds the A rows of M-tile r and the B columns of output
// channels 32r .. 32r+31 of every x tap (its half of dY, staged with 64-byte
// swizzle so that the X atoms of 32 columns sit one dil_w pixel row apart, as
// the 64-column atoms of the single-CTA form do).  Per SM and K-step the
// operand reads fall to 4 KB + 16*N bytes and the TMA writes to one X patch
// plus half a dY patch.  Rank r's TMEM holds rows of M-tile r, columns ordered
// (k half, x block, k): column 32*X*h + 32*j + kk is k = 32h + kk of tap
// x = X-1-j.
//
// Both CTAs load the same X box (the two requests reach L2 together, as the
// two single-CTA M-ranges of a split do); one A descriptor serves the pair
// because rank 1 places its copy pair_xshift bytes (its first atom's row
// offset) lower in the stage: stage = [dY half][pair_xshift][X patch] for
// rank 0, [dY half][X patch][pair_xshift] for rank 1, whose padding atom (the
// fourth, when the filter has three rows) reads into its own tail.  A box that
// is shifted down instead measured ~20% more L2 sectors and a slower loop.
//
// Barriers: rank 0's full[stage] counts both CTAs' TMA bytes (rank 1's loads
// signal it across the pair); rank 0's MMA commits arrive on empty[stage] and
// on the accumulator barrier of both CTAs.  Every wait is bounded; both CTAs
// pass two cluster barriers (barriers initialised and TMEM allocated; before
// releasing TMEM) on every path.
#pragma once

#include "k_igemm.cuh"

namespace wg {

__global__ void __launch_bounds__(kIgThreads, 1)
    igemm_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                            const __grid_constant__ IgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_shared<uint8_t>(smem_raw, 1024);
    // [stages x stage_bytes][1 KB slack][tail: barriers + TMEM address]
    uint8_t* tail = smem + p.stages * p.stage_bytes + 1024;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);
    uint64_t* empty = full + 8;
    uint64_t* accb = empty + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);

    // The host launches this kernel only for pair plans (uniform over the grid,
    // so no CTA waits at a cluster barrier for one that returned here).
    if (!p.pair || !p.xs || p.mtpc != 1 || p.n_mtiles != 2 || p.ncc != 1 || p.staged || p.clq != 1 ||
        gridDim.x != 2) {
        if (threadIdx.x == 0) atomicOr(&g_status, kStatusBadPlan);
        return;
    }
    const int ksteps = p.ksteps, stages = p.stages, stage_bytes = p.stage_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();  // = blockIdx.x: M-tile of this CTA
    const int gb = blockIdx.y, split = blockIdx.z;
    const int kt0 = split * p.per_split;
    const int nk = max(0, min(p.per_split, p.total_kt - kt0));
    const int g0 = gb * p.Gm;
    const int c_al = (g0 * p.C) & ~7;
    const int k_base = (g0 * p.K) & ~7;

    pdl_launch_dependents();
    // Stage i: the X patch (the same box in both CTAs; rank 1's copy
    // pair_xshift bytes lower) and this CTA's 32 channels of the dY patch; the
    // bytes are counted on rank 0's full[stage], which expects both CTAs' loads.
    const uint32_t tx_cta = (uint32_t)(p.patch_tx + p.dy_tx);
    const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0u);
    const int xoff = p.pair_xoff - rank * p.pair_xshift;
    auto issue_stage = [&](int i) {
        const int st = i % stages;
        uint8_t* sb = smem + st * stage_bytes;
        if (rank == 0) mbar_arrive_expect_tx(&full[st], 2u * tx_cta);
        int kt = kt0 + i;
        const int tw = kt % p.ntile[0];
        kt /= p.ntile[0];
        const int th = kt % p.ntile[1];
        kt /= p.ntile[1];
        const int td = kt % p.ntile[2];
        const int tn = kt / p.ntile[2];
        const int wo0 = tw * p.box[0], ho0 = th * p.box[1], do0 = td * p.box[2], n0 = tn * p.box[3];
        const uint32_t bar = full0 + (uint32_t)(st * 8);
        tma_load_5d_pair(sb + xoff, &tmx, bar, c_al, wo0 - p.pl[0] + p.patch_ph[0][0], ho0 - p.pl[1] + p.patch_ph[0][1],
                         do0 - p.pl[2] + p.patch_ph[0][2], n0);
        tma_load_5d_pair(sb + p.dy_off, &tmy, bar, k_base + 32 * rank, wo0 - p.dy_xoff, ho0, do0, n0);
    };
    const bool wait_first = p.mode != 2;
    if (threadIdx.x == 0) {
        if (nk > 0) {
            tma_prefetch_desc(&tmx);
            tma_prefetch_desc(&tmy);
        }
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accb, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        // TMEM may still be held by the kernel before this one until it completes.
        if (wait_first) pdl_wait();
        tmem_alloc_pair(tslot, (uint32_t)p.tmem_cols);
        tc_fence_before();
    }
    // One cluster barrier: past it, both CTAs' barriers are initialised (rank
    // 1's loads signal rank 0's) and both hold their TMEM (rank 0's MMAs write
    // both).  Rank 0 sends its first stage between arriving and waiting, to its
    // own barrier; rank 1 sends its first stage after the wait.  (Issuing every
    // ring stage up front put all of the call's input in flight at once: each
    // CTA's first stage then landed ~1 us later.)
    cluster_arrive();
    int pre = 0;
    if (threadIdx.x == 0 && nk > 0 && rank == 0) {
        if (wait_first) pdl_wait();
        pre = 1;
        issue_stage(0);
    }
    cluster_wait();
    if (threadIdx.x == 0 && nk > 0 && rank == 1) {
        if (wait_first) pdl_wait();
        pre = 1;
        issue_stage(0);
    }
    tc_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == 0) {
        if (lane == 0 && nk > 0) {
            // ------------------------------------------------ TMA producer (each CTA)
            for (int i = pre; i < nk; ++i) {
                const int st = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (i >= stages && !mbar_wait(&empty[st], ph ^ 1u)) break;
                issue_stage(i);
            }
        }
    } else if (warp == 1) {
        if (rank == 0 && nk > 0) {
            // ------------------------------------------------ MMA issuer (rank 0, whole warp)
            // A: the two atoms of the CTA's M-tile (rank 1's patch copy is placed
            // so that its atoms sit at the same offsets); B: X atoms of 32
            // columns, one dil_w row apart, 64-byte swizzle.
            const uint32_t sbase = smem_u32(smem);
            const uint64_t a0 =
                make_sdesc(sbase + (uint32_t)p.pair_xoff + p.atom_off[0], p.atom_off[1] - p.atom_off[0], 0u, 2u, 0u);
            const uint64_t b0 = make_sdesc(sbase + (uint32_t)p.dy_off, (uint32_t)(p.d[0] * 64), 0u, 4u, 0u);
            const uint32_t idesc = p.idesc, stage16 = (uint32_t)stage_bytes >> 4;
            int st = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nk; ++i) {
                if (!mbar_wait(&full[st], ph)) break;
                tc_fence_after();
                const uint64_t soff = (uint64_t)((uint32_t)st * stage16);
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {
                    if (ks >= ksteps) break;
                    const uint64_t ad = a0 + p.kd_table[ks] + soff;
                    const uint64_t bd = b0 + p.kd_table_b[ks] + soff;
                    const uint32_t acc = (i | ks) != 0 ? 1u : 0u;
                    if (elect_one()) umma_f16_pair(tbase, ad, bd, idesc, acc);
                    __syncwarp();
                }
                if (elect_one()) umma_commit_pair(&empty[st]);
                __syncwarp();
                if (++st == stages) st = 0, ph ^= 1u;
            }
            if (elect_one()) umma_commit_pair(accb);
            __syncwarp();
        }
    }
    __syncwarp();
    // ---------------------------------------------------- epilogue (all warps, both CTAs)
    named_bar_sync(2, kIgThreads);
    // Atomic mode: dW was zeroed by the kernel this one depends on; every
    // thread passes the wait before its first global write.
    pdl_wait();
    if (nk > 0) {
        mbar_wait_sleep(accb, 0);
        tc_fence_after();
    }
    {
        const int q = warp & 3, h = warp >> 2;
        const int row = q * 32 + lane;
        const int K = p.K, C = p.C, T = p.T, xs = p.xs, mode = p.mode, out_dtype = p.out_dtype;
        void* const out = p.out;
        const uint32_t trow = tbase + ((uint32_t)(q * 32) << 16);
        const bool have_acc = nk > 0;
        const int atom = 2 * rank + (row >> 6);
        bool vrow = atom < p.n_atoms;
        const int tap = vrow ? p.atom_tap[atom] : 0;  // tap of x = 0
        const int cg = c_al + (row & 63);
        const int gr = cg / C;
        const int c = cg - gr * C;
        vrow = vrow && cg < p.GC && gr >= g0 && gr < g0 + p.Gm;
        // Columns of this warp: k half h, 32 per x block; k = 32h + column - 32*(xs*h + j).
        const int nl = gr * K - k_base - 32 * h;
        const long long kstride = (long long)T * C;
        for (int j = 0; j < xs; ++j) {
            const int tapj = tap + (xs - 1 - j);
            const uint32_t ta = trow + (uint32_t)(32 * (xs * h + j));
            const long long rowbase = ((long long)gr * K * T + tapj) * C + c;
            if (mode == 3) {
                const long long x = (long long)tapj * C + c;
                const long long jj = x / p.ws.W;
                const long long wbase =
                    (((long long)gr * K * p.ws.nj + jj) * p.ws.S + split) * p.ws.W + (x - jj * p.ws.W);
                epilogue_mtile<3, float>(ta, 32, have_acc, vrow, nl, K, static_cast<float*>(out), wbase,
                                         (long long)p.ws.nj * p.ws.S * p.ws.W);
            } else if (mode == 2) {
                if (have_acc)
                    epilogue_mtile<2, float>(ta, 32, true, vrow, nl, K, static_cast<float*>(out), rowbase, kstride);
            } else if (out_dtype == 2) {
                epilogue_mtile<1, float>(ta, 32, have_acc, vrow, nl, K, static_cast<float*>(out), rowbase, kstride);
            } else if (out_dtype == 0) {
                epilogue_mtile<1, __nv_bfloat16>(ta, 32, have_acc, vrow, nl, K, static_cast<__nv_bfloat16*>(out),
                                                 rowbase, kstride);
            } else {
                epilogue_mtile<1, __half>(ta, 32, have_acc, vrow, nl, K, static_cast<__half*>(out), rowbase,
                                          kstride);
            }
        }
    }
    // Neither CTA releases TMEM or leaves while the pair's MMAs or loads may
    // still touch the other's memory.
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tbase, (uint32_t)p.tmem_cols);
    }
}

}  // namespace wg
