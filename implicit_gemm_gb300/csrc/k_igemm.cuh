// Tensor-core implicit-GEMM weight gradient (sm_103a: TMA + tcgen05 + TMEM).
//
// The GEMM of "Composable Kernel: grouped_convolution_backward_weight_kernel.hpp
// Source File" (GroupedConvBwdWeightKernelArgs: GemmM = K, GemmN = C*YX,
// GemmK = N*Ho*Wo, batched over G via the group strides; grid = (tiles, G,
// k_batch) in GridSize / operator()) is computed here as its transpose
//
//     D[(tap, c), k] = sum over pixels p of Xcol[p, (tap, c)] * dY[p, k]
//
// so that the long (tap, c) axis sits on the 128 MMA rows and the output
// channels k on the MMA N columns.  Both operands are staged in shared memory
// with the free axis contiguous and the reduction axis (pixels) strided -- the
// "K-outer" arrangement that PR #11602 ("add transpose load for bwd weight and
// bwd data") describes for gfx950 -- which tcgen05 consumes directly as
// MN-major operands (128-byte swizzle), so nothing is ever transposed.
//
// X staging (chosen by the planner):
//  * halo: one TMA box per (stride phase, 64-channel chunk) covers every tap
//    of a K-tile of output pixels; the A operand of tap (z,y,x) is the same
//    patch read from a row offset (shared-memory descriptors are
//    address-swizzled, so any 128-byte row offset is a valid start).
//  * per-tap: one TMA box per (tap, chunk) with the tap offset in its
//    coordinates and the conv stride as the TMA element stride.
// Implicit zero padding is the TMA out-of-bounds fill, for both operands.
//
// Tap forms.  With every tap on the rows, K = 64 output channels give N = 64,
// and a 128x64x16 MMA is bound by its shared-memory operand reads.  For
// stride 1 the pixel sum can run over q = wo + x*dil_w instead, with dY read
// at q - x*dil_w (zero outside the image) and X at q - pad: the x taps then
// sit on the columns, D[(z, y, c), (x, k)], B being one dY patch per K-tile
// read as xs 64-column atoms one dil_w row apart -- 128x192x16 MMAs for 3x3
// filters, at the tensor rate.
//
// Warp roles (256 threads): warp 0 lane 0 issues TMA; warp 1 owns TMEM and, as
// a converged warp, issues tcgen05.mma from one elected lane; after the main
// loop all eight warps read TMEM (lane quadrant = warp % 4, column half =
// warp / 4) and store dW / atomically add / write the split-K workspace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"

namespace wg {

// Most M-tiles one CTA accumulates (TMEM columns = M-tiles x Nt <= 512).
constexpr int kMaxMt = 16;

// Threads of igemm_wgrad_kernel: warp 0 lane 0 issues the TMA loads, warp 1
// the MMAs; after the main loop all eight warps read the accumulators out of
// TMEM (warp w reads lane quadrant w % 4, columns of half w / 4).
constexpr int kIgThreads = 256;

struct IgParams {
    int G, C, K, T, GC, GK;
    int X, Y;                // filter extents along w and h (tap = (z*Y + y)*X + x)
    int ncc;                 // 64-channel chunks per tap
    int s[3], d[3], pl[3];   // stride, dilation, left pad along (w, h, d)
    int box[4], ntile[4];    // pixel tile and tile counts along (w, h, d, n)
    int KT, ksteps;
    int per_split, total_kt;
    int Gm, Nt, n_ntiles, n_katoms, n_atoms, n_mtiles, mtpc;
    int halo;
    // Tap form: xs = 0, every tap on the MMA rows; xs = X, the x taps on the
    // columns (atoms are (z, y, chunk); B atom j = tap x = xs-1-j of one dY
    // patch per K-tile, dy_xoff = (X-1)*dil_w columns of it left of the tile).
    int xs, Nmma, dy_tx, dy_xoff;
    int patch[3];
    int patch_bytes, patch_tx;
    int n_patches, dy_off, slot_bytes, stage_bytes, stages;
    int tmem_cols;
    uint32_t idesc;
    int mode;       // 1 direct, 2 atomic, 3 workspace
    int out_dtype;  // wg_dtype
    int clq;        // CTAs per cluster along the split (1: no cluster reduction)
    // Staged output (split modes): the CTA covers whole groups (every tap,
    // channel and k of groups g0 .. g0 + Gm - 1, windows starting at their first
    // channel), so its results form one contiguous block of dW, Gm*K*T*C
    // elements, that the epilogue gathers in shared memory and adds or stores
    // with 16-byte accesses.
    int staged;
    // CTA pair (igemm_wgrad_pair_kernel): the split's two M-tiles run on the
    // two CTAs of a cluster that share M = 256 MMAs.  Both load the same X
    // patch, rank 0 at byte pair_xoff of the stage and rank 1 pair_xshift
    // bytes lower, so that rank 1's first atom (the tile's third) sits at the
    // offset of rank 0's first atom.
    int pair, pair_xoff, pair_xshift;
    // Staged output: atom_of[(tap / (xs ? xs : 1)) * ncc + cc] is the index of
    // the atom holding channel chunk cc of filter tap `tap` (x = 0 when the x
    // taps sit on the columns).
    unsigned char atom_of[256];
    void* out;
    WsLayout ws;    // split-K workspace layout (mode 3): rows (g, k) of L = T * C, S / clq partials
    unsigned char patch_ph[32][4];
    unsigned int atom_off[256];
    unsigned short atom_tap[256];
    unsigned char atom_cc[256];
    // K-step part of the A descriptor, the same for every K-tile: row offset of
    // the step's first 8-pixel group (start-address field) and the byte offset
    // of its second group (SBO field).  Filled on the host.
    unsigned long long kd_table[16];
    // The same for the B operand when xs > 0 (rows of the dY patch).
    unsigned long long kd_table_b[16];
};

// Up to kEpiCols consecutive TMEM columns (n a multiple of 16) with one wait:
// the loads are issued back to back, so their latencies overlap.
constexpr int kEpiCols = 32;
__device__ __forceinline__ void tmem_ld_batch(uint32_t taddr, int n, float (&v)[kEpiCols])
{
    uint32_t r[kEpiCols];
#pragma unroll
    for (int q = 0; q < kEpiCols / 16; ++q)
        if (16 * q < n) tmem_ld16_issue(taddr + (uint32_t)(16 * q), r + 16 * q);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int q = 0; q < kEpiCols / 16; ++q)
        if (16 * q < n) reg_fence16(r + 16 * q);
#pragma unroll
    for (int i = 0; i < kEpiCols; ++i) v[i] = __uint_as_float(r[i]);
}

// Epilogue of one M-tile for one warp: TMEM -> registers -> global, in chunks
// of up to kEpiCols columns.  MODE 1 stores dW in OUT (fp32, bf16 or fp16), MODE 2
// adds to fp32 dW with global atomics, MODE 3 stores fp32 to the split's
// workspace slice.  Each lane owns one row (tap, c); k runs over the columns,
// so a warp's store covers 32 consecutive channels.
template <int MODE, typename OUT>
__device__ __forceinline__ void epilogue_mtile(uint32_t taddr, int ncols, bool have_acc, bool vrow, int n_lo, int K,
                                               OUT* __restrict__ out, long long rowbase, long long kstride)
{
    for (int cb = 0; cb < ncols; cb += kEpiCols) {
        const int n = min(kEpiCols, ncols - cb);
        float v[kEpiCols];
        if (have_acc) {
            tmem_ld_batch(taddr + (uint32_t)cb, n, v);
        } else {
#pragma unroll
            for (int j = 0; j < kEpiCols; ++j) v[j] = 0.f;
        }
        if (!vrow) continue;
        const int k0 = cb - n_lo;
        OUT* o = out + rowbase + (long long)k0 * kstride;
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) {
            const int k = k0 + j;
            if (j < n && k >= 0 && k < K) {
                if constexpr (MODE == 2) {
                    red_add_f32(reinterpret_cast<float*>(o), v[j]);
                } else if constexpr (sizeof(OUT) == 4) {
                    *o = v[j];
                } else if constexpr (sizeof(OUT) == 2 && std::is_same<OUT, __nv_bfloat16>::value) {
                    *o = __float2bfloat16_rn(v[j]);
                } else {
                    *o = __float2half_rn(v[j]);
                }
            }
            o += kstride;
        }
    }
}

// Store one output element of row `row` (a (tap, channel) pair of the CTA's
// window) and column `col` (a k of the CTA's N-tile) in the epilogue's mode.
struct RowMap {
    long long base;  // dW index of (group, k = 0, tap, c); < 0: row outside the window
    int n_lo;        // column of k = 0 of the row's group
};

__device__ __forceinline__ RowMap map_row(const IgParams& p, int atom, int row64, int c_al, int g0, int k_base)
{
    RowMap r{-1, 0};
    if (atom >= p.n_atoms) return r;
    int tap, cc;
    if (p.halo) {
        tap = p.atom_tap[atom];
        cc = p.atom_cc[atom];
    } else {
        tap = atom / p.ncc;
        cc = atom - tap * p.ncc;
    }
    const int cg = c_al + cc * 64 + row64;
    const int gr = cg / p.C;
    const int c = cg - gr * p.C;
    if (cg >= p.GC || gr < g0 || gr >= g0 + p.Gm) return r;
    r.base = ((long long)gr * p.K * p.T + tap) * p.C + c;
    r.n_lo = gr * p.K - k_base;
    return r;
}

__device__ __forceinline__ void store_elem(int mode, int out_dtype, void* out, long long i, float v,
                                           const WsLayout& ws, int ws_s)
{
    if (mode == 2) {
        red_add_f32(static_cast<float*>(out) + i, v);
    } else if (mode == 3) {
        static_cast<float*>(out)[ws_offset(ws, i, ws_s)] = v;
    } else if (out_dtype == 2) {
        static_cast<float*>(out)[i] = v;
    } else if (out_dtype == 0) {
        static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half*>(out)[i] = __float2half_rn(v);
    }
}

// Cluster reduction of the split-K partial sums, run by the eight warps of
// every CTA of a cluster once each CTA has staged its accumulators in
// its own shared memory, column-major (red[(m * Nt + col) * 128 + row]).  The
// mtn * Nt columns are dealt out to the cluster's CTAs in contiguous ranges;
// for each of its columns a warp reads the 128 rows (lane = rows lane,
// lane + 32, lane + 64, lane + 96) from every CTA of the cluster through
// distributed shared memory, adds them in rank order -- a fixed order, so the
// result is reproducible -- and stores the sums (the dW values, or the
// cluster's partial sums) as whole 128-byte rows of consecutive channels.
__device__ __forceinline__ void cluster_reduce_store(const IgParams& p, uint32_t red_s, int mtn, int atom0, int c_al,
                                                     int g0, int k_base, void* out, int ws_s, int ew, int lane)
{
    const int Q = p.clq, Nt = p.Nt, K = p.K, mode = p.mode, out_dtype = p.out_dtype;
    const long long kstride = (long long)p.T * p.C;
    const int rank = (int)cluster_ctarank();
    const int U = mtn * Nt;
    const int u0 = (int)((long long)U * rank / Q), u1 = (int)((long long)U * (rank + 1) / Q);
    uint32_t peer[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) peer[r] = r < Q ? mapa_shared(red_s, (uint32_t)r) : 0u;
    int m_cur = -1;
    RowMap rm[4];
    for (int u = u0 + ew; u < u1; u += kIgThreads / 32) {
        float v[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (r < Q) {
#pragma unroll
                for (int i = 0; i < 4; ++i) v[r][i] = ld_dsmem_f32(peer[r] + (uint32_t)(u * 128 + 32 * i + lane) * 4u);
            }
        const int m = u / Nt, col = u - m * Nt;
        if (m != m_cur) {
            m_cur = m;
#pragma unroll
            for (int i = 0; i < 4; ++i) rm[i] = map_row(p, atom0 + 2 * m + (i >> 1), (32 * i + lane) & 63, c_al, g0, k_base);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float a = v[0][i];
#pragma unroll
            for (int r = 1; r < 8; ++r)
                if (r < Q) a += v[r][i];
            const int k = col - rm[i].n_lo;
            if (rm[i].base >= 0 && k >= 0 && k < K)
                store_elem(mode, out_dtype, out, rm[i].base + k * kstride, a, p.ws, ws_s);
        }
    }
}

struct MmaArgs {
    uint64_t b0;        // dY descriptor of stage 0, K-step 0
    uint32_t idesc, Nt, stage16;  // Nt: TMEM columns per M-tile (the MMA N)
    int ksteps, stages;
};

// The MMA issuer, run by a whole converged warp; one elected lane issues a
// K-step's MT MMAs.  Every operand is a sum of 64-bit parts whose fields never
// overlap: the M-tile part ab[m] (start of its first atom in stage 0, LBO to
// its second atom), the K-step part kdt[ks] (from the kernel parameters) and
// the stage offset.  The K-step loop is unrolled against the parameter table:
// descriptor operands built from runtime geometry inside the loop halved the
// MMA issue rate.
template <int MT, bool XS>
__device__ __forceinline__ void mma_mainloop(const MmaArgs a, const uint64_t (&ab)[kMaxMt], uint64_t* full,
                                             uint64_t* empty, uint64_t* accb, uint32_t tbase, int nk,
                                             const unsigned long long* __restrict__ kdt,
                                             const unsigned long long* __restrict__ kdtb)
{
    const uint64_t b0 = a.b0;
    const uint32_t idesc = a.idesc, Nt = a.Nt, stage16 = a.stage16;
    const int ksteps = a.ksteps, stages = a.stages;
    int st = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nk; ++i) {
        if (!mbar_wait(&full[st], ph)) break;
        tc_fence_after();
        const uint64_t soff = (uint64_t)((uint32_t)st * stage16);
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
            if (ks >= ksteps) break;
            const uint64_t kd = kdt[ks] + soff;
            const uint64_t bdesc = XS ? b0 + soff + kdtb[ks] : b0 + soff + (uint64_t)(ks * 128);
            const uint32_t acc = (i | ks) != 0 ? 1u : 0u;
            if (elect_one()) {
#pragma unroll
                for (int m = 0; m < MT; ++m) umma_f16(tbase + (uint32_t)m * Nt, ab[m] + kd, bdesc, idesc, acc);
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(&empty[st]);
        __syncwarp();
        if (++st == stages) st = 0, ph ^= 1u;
    }
    if (elect_one()) umma_commit(accb);
    __syncwarp();
}

// SPEC 0 handles every plan.  SPEC 1 is the same kernel compiled for one plan
// family only -- the x taps on the MMA columns, one M-tile per CTA, a split
// mode (atomic or two-stage) -- without the other MMA loop instances and the
// direct-store epilogue: the smaller kernel runs the 56x56 C = K = 64 workload
// in 15.3-15.5 us per call against 16.3 us for the general one (the other
// workloads, which use other plan families, measured no gain from trimming).
template <int SPEC>
__global__ void __launch_bounds__(kIgThreads, 1)
    igemm_wgrad_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                       const __grid_constant__ IgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_shared<uint8_t>(smem_raw, 1024);
    // [stages x stage_bytes][1 KB slack read by padding atoms][tail: barriers + tables]
    uint8_t* tail = smem + p.stages * p.stage_bytes + 1024;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);
    uint64_t* empty = full + 8;
    uint64_t* accb = empty + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);

    if constexpr (SPEC == 1) {
        // The host launches this instance only for its plan family.
        if (!p.xs || p.mtpc != 1 || p.mode == 1 || p.pair) {
            if (threadIdx.x == 0) atomicOr(&g_status, kStatusBadPlan);
            return;
        }
    } else {
        // Pair plans run on igemm_wgrad_pair_kernel.
        if (p.pair) {
            if (threadIdx.x == 0) atomicOr(&g_status, kStatusBadPlan);
            return;
        }
    }
    // Scalars used in loops are read into registers once here.
    const int Nt = p.Nt, ksteps = p.ksteps, stages = p.stages, stage_bytes = p.stage_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mr = blockIdx.x / p.n_ntiles, nt = blockIdx.x % p.n_ntiles;
    const int gb = blockIdx.y, split = blockIdx.z;
    const int kt0 = split * p.per_split;
    const int nk = max(0, min(p.per_split, p.total_kt - kt0));
    const int mt0 = mr * p.mtpc;
    const int mtn = min(p.mtpc, p.n_mtiles - mt0);
    const int atom0 = 2 * mt0;
    const int g0 = gb * p.Gm;
    const int c_al = (g0 * p.C) & ~7;
    const int k_base = ((g0 * p.K) & ~7) + nt * p.Nt;

    // The kernel launched after this one (the split reduction, or the next
    // call's first kernel) may be scheduled at once; it waits for this whole
    // grid's results before it reads them.
    pdl_launch_dependents();
    // Stage i of the TMA ring: the K-tile's X patches (or per-tap boxes) and dY.
    const uint32_t tx = (uint32_t)(p.n_patches * p.patch_tx + p.dy_tx);
    auto issue_stage = [&](int i) {
        const int st = i % p.stages;
        uint8_t* sb = smem + st * p.stage_bytes;
        mbar_arrive_expect_tx(&full[st], tx);
        int kt = kt0 + i;
        const int tw = kt % p.ntile[0];
        kt /= p.ntile[0];
        const int th = kt % p.ntile[1];
        kt /= p.ntile[1];
        const int td = kt % p.ntile[2];
        const int tn = kt / p.ntile[2];
        const int wo0 = tw * p.box[0], ho0 = th * p.box[1], do0 = td * p.box[2], n0 = tn * p.box[3];
        const int bw = wo0 * p.s[0] - p.pl[0], bh = ho0 * p.s[1] - p.pl[1], bd = do0 * p.s[2] - p.pl[2];
        if (p.halo) {
            for (int q = 0; q < p.n_patches; ++q)
                tma_load_5d(sb + q * p.patch_bytes, &tmx, &full[st], c_al + 64 * p.patch_ph[q][3],
                            bw + p.patch_ph[q][0], bh + p.patch_ph[q][1], bd + p.patch_ph[q][2], n0);
        } else {
            for (int a = 0; a < p.n_patches; ++a) {
                const int atom = atom0 + a;
                if (a < 2 * mtn && atom < p.n_atoms) {
                    const int tap = atom / p.ncc, cc = atom - tap * p.ncc;
                    const int x = tap % p.X, y = (tap / p.X) % p.Y, z = tap / (p.X * p.Y);
                    tma_load_5d(sb + a * p.patch_bytes, &tmx, &full[st], c_al + 64 * cc, bw + x * p.d[0],
                                bh + y * p.d[1], bd + z * p.d[2], n0);
                } else {
                    // Padding atom: a box entirely past the channel extent reads zeros.
                    tma_load_5d(sb + a * p.patch_bytes, &tmx, &full[st], p.GC, 0, 0, 0, 0);
                }
            }
        }
        for (int j = 0; j < p.n_katoms; ++j)
            tma_load_5d(sb + p.dy_off + j * p.slot_bytes, &tmy, &full[st], k_base + 64 * j, wo0 - p.dy_xoff,
                        ho0, do0, n0);
    };
    // Thread 0 (the TMA producer) initialises the barriers and issues the first
    // stage before the block barrier, and warp 1 allocates TMEM meanwhile: the
    // tensor maps' first fetch by the TMA unit (~1 us) then overlaps the
    // prologue instead of following it.  (Issuing every ring stage here held
    // the other warps at the barrier for longer than the data took to land.)
    // This kernel is a programmatic dependent of the kernel before it on the
    // stream.  Unless that kernel is this call's zeroing kernel (which itself
    // waited for everything before it), X and dY are read only after
    // griddepcontrol.wait, and so is TMEM taken (a kernel before it could still
    // be about to allocate); the tensor-map prefetch and the barrier set-up run
    // before, overlapping the previous kernel's tail.
    const bool wait_first = p.mode != 2;
    int pre = 0;
    if (threadIdx.x == 0) {
        if (nk > 0) {
            tma_prefetch_desc(&tmx);
            tma_prefetch_desc(&tmy);
        }
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accb, 1);
        fence_mbar_init();
        if (wait_first) pdl_wait();
        pre = min(1, nk);
        for (int i = 0; i < pre; ++i) issue_stage(i);
    }
    if (warp == 1) {
        if (wait_first) pdl_wait();
        tmem_alloc(tslot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();  // barriers initialised, TMEM allocated, the first stage on its way
    // The producer reads the TMEM address after the main loop.
    uint32_t tbase = 0;
    if (warp != 0) {
        tc_fence_after();
        tbase = *tslot;
    }
#define MMA_ARGS ma, ab, full, empty, accb, tbase, nk, p.kd_table, p.kd_table_b

    if (warp == 0) {
        if (lane == 0 && nk > 0) {
            // ------------------------------------------------ TMA producer
            for (int i = pre; i < nk; ++i) {
                const int st = i % p.stages;
                const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
                if (i >= p.stages && !mbar_wait(&empty[st], ph ^ 1u)) break;
                issue_stage(i);
            }
        }
    } else if (warp == 1) {
        if (nk > 0) {
            // ------------------------------------------------ MMA issuer (whole warp)
            const uint32_t sbase = smem_u32(smem);
            uint64_t ab[kMaxMt];
#pragma unroll
            for (int m = 0; m < kMaxMt; ++m) {
                ab[m] = 0;
                if (m < mtn) {
                    const int a = atom0 + 2 * m;
                    uint32_t off_a, off_b;
                    if (p.halo) {
                        off_a = p.atom_off[a];
                        off_b = (a + 1 < p.n_atoms) ? p.atom_off[a + 1] : off_a + 1024u;
                    } else {
                        off_a = (uint32_t)(2 * m * p.patch_bytes);
                        off_b = off_a + (uint32_t)p.patch_bytes;
                    }
                    ab[m] = make_sdesc(sbase + off_a, off_b - off_a, 0u, 2u, 0u);
                }
            }
            MmaArgs ma;
            ma.idesc = p.idesc, ma.Nt = (uint32_t)p.Nmma, ma.stage16 = (uint32_t)stage_bytes >> 4;
            ma.ksteps = ksteps, ma.stages = stages;
            if (p.xs) {
                // One dY patch: B atom j starts j*dil_w rows in (LBO); the K-step
                // part (start row, SBO) comes from kd_table_b.
                ma.b0 = make_sdesc(sbase + (uint32_t)p.dy_off, (uint32_t)(p.d[0] * 128), 0u, 2u, 0u);
                if constexpr (SPEC == 1) {
                    mma_mainloop<1, true>(MMA_ARGS);
                } else {
                    switch (mtn) {
                        case 1: mma_mainloop<1, true>(MMA_ARGS); break;
                        case 2: mma_mainloop<2, true>(MMA_ARGS); break;
                        case 3: mma_mainloop<3, true>(MMA_ARGS); break;
                        default: mma_mainloop<4, true>(MMA_ARGS); break;
                    }
                }
            } else if constexpr (SPEC == 0) {
                ma.b0 = make_sdesc(sbase + (uint32_t)p.dy_off, (uint32_t)p.slot_bytes, 1024u, 2u, 0u);
                switch (mtn) {
                    case 1: mma_mainloop<1, false>(MMA_ARGS); break;
                    case 2: mma_mainloop<2, false>(MMA_ARGS); break;
                    case 3: mma_mainloop<3, false>(MMA_ARGS); break;
                    case 4: mma_mainloop<4, false>(MMA_ARGS); break;
                    case 5: mma_mainloop<5, false>(MMA_ARGS); break;
                    case 6: mma_mainloop<6, false>(MMA_ARGS); break;
                    case 7: mma_mainloop<7, false>(MMA_ARGS); break;
                    case 8: mma_mainloop<8, false>(MMA_ARGS); break;
                    case 9: mma_mainloop<9, false>(MMA_ARGS); break;
                    case 10: mma_mainloop<10, false>(MMA_ARGS); break;
                    case 11: mma_mainloop<11, false>(MMA_ARGS); break;
                    case 12: mma_mainloop<12, false>(MMA_ARGS); break;
                    case 13: mma_mainloop<13, false>(MMA_ARGS); break;
                    case 14: mma_mainloop<14, false>(MMA_ARGS); break;
                    case 15: mma_mainloop<15, false>(MMA_ARGS); break;
                    default: mma_mainloop<16, false>(MMA_ARGS); break;
                }
            }
        }
    }
    __syncwarp();
    // ---------------------------------------------------- epilogue (all warps)
    named_bar_sync(2, kIgThreads);  // the producer is done and may read tbase
    // Atomic accumulation: dW was zeroed by a kernel launched just before this
    // one (programmatic dependent launch); wait for it only here, so that its
    // launch and run overlap the main loop.  In the other modes the previous
    // kernel finished before the first stage was loaded and this returns at
    // once; every thread passes it before its first global write.
    pdl_wait();
    tc_fence_after();
    tbase = *tslot;
    {
        if (nk > 0) {
            mbar_wait_sleep(accb, 0);
            tc_fence_after();
        }
        const int q = warp & 3;
        const int row = q * 32 + lane;
        // Column half of this warp: [c_lo, c_hi) of the MMA N, split at a multiple of 16.
        const int Nmma = p.Nmma;
        const int c_mid = ((Nmma >> 1) + 15) & ~15;
        const int c_lo = warp < 4 ? 0 : c_mid, c_hi = warp < 4 ? c_mid : Nmma;
        const int K = p.K, C = p.C, T = p.T, GC = p.GC, Gm = p.Gm, n_atoms = p.n_atoms, ncc = p.ncc, mode = p.mode;
        const int out_dtype = p.out_dtype;
        void* const out = p.out;
        const int ws_s = split / p.clq;
        const uint32_t trow = tbase + ((uint32_t)(q * 32) << 16);
        const bool have_acc = nk > 0;
        if (p.clq > 1) {
            // Stage the accumulators for the cluster reduction in the (now idle)
            // pipeline buffers, column-major so that a warp's stores are
            // consecutive words.
            float* red = reinterpret_cast<float*>(smem);
            for (int m = 0; m < mtn; ++m)
                for (int cb = c_lo; cb < c_hi; cb += kEpiCols) {
                    const int n = min(kEpiCols, c_hi - cb);
                    float v[kEpiCols];
                    if (have_acc) {
                        tmem_ld_batch(trow + (uint32_t)(m * Nt + cb), n, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < kEpiCols; ++j) v[j] = 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < kEpiCols; ++j)
                        if (j < n) red[(m * Nt + cb + j) * 128 + row] = v[j];
                }
        }
        if (p.staged) {
            // Dump the accumulators into the idle pipeline buffers column by
            // column (dump[(m * Nmma + col) * 128 + row]: a warp's 32 rows of a
            // column are 32 consecutive words); the valid (diagonal) elements
            // are picked out in dW order after the barrier below.
            float* dump = reinterpret_cast<float*>(smem);
            for (int m = 0; m < mtn; ++m)
                for (int cb = c_lo; cb < c_hi; cb += kEpiCols) {
                    const int n = min(kEpiCols, c_hi - cb);
                    float v[kEpiCols];
                    if (have_acc) {
                        tmem_ld_batch(trow + (uint32_t)(m * Nmma + cb), n, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < kEpiCols; ++j) v[j] = 0.f;
                    }
                    float* d = dump + (m * Nmma + cb) * 128 + row;
#pragma unroll
                    for (int j = 0; j < kEpiCols; ++j)
                        if (j < n) d[j * 128] = v[j];
                }
        }
        for (int m = 0; m < mtn && p.clq == 1 && !p.staged; ++m) {
            const int atom = atom0 + 2 * m + (row >> 6);
            bool vrow = atom < n_atoms;
            int tap = 0, cc = 0;
            if (vrow) {
                if (p.halo) {
                    tap = p.atom_tap[atom];
                    cc = p.atom_cc[atom];
                } else {
                    tap = atom / ncc;
                    cc = atom - tap * ncc;
                }
            }
            const int cg = c_al + cc * 64 + (row & 63);
            const int gr = cg / C;
            const int c = cg - gr * C;
            vrow = vrow && cg < GC && gr >= g0 && gr < g0 + Gm;
            const int n_lo = gr * K - k_base;
            const long long kstride = (long long)T * C;
            // Column blocks: the whole N-tile, or with the x taps on the
            // columns one 64-column block per tap x = xs-1-jb (the atom's tap
            // entry is that of x = 0).
            const int nblk = p.xs ? p.xs : 1, bw = p.xs ? 64 : Nmma;
            for (int jb = 0; jb < nblk; ++jb) {
                const int lo = max(c_lo, jb * bw), hi = min(c_hi, jb * bw + bw);
                if (lo >= hi) continue;
                const int tapj = p.xs ? tap + (p.xs - 1 - jb) : tap;
                const long long rowbase = ((long long)gr * K * T + tapj) * C + c;
                const uint32_t ta = trow + (uint32_t)(m * Nmma + lo);
                const int nc = hi - lo, nl = n_lo - (lo - jb * bw);
                if (mode == 3) {
                    // Workspace: the row's first element (k = 0) and the step per k.
                    const long long x = (long long)tapj * C + c;
                    const long long j = x / p.ws.W;
                    const long long wbase =
                        (((long long)gr * K * p.ws.nj + j) * p.ws.S + ws_s) * p.ws.W + (x - j * p.ws.W);
                    epilogue_mtile<3, float>(ta, nc, have_acc, vrow, nl, K, static_cast<float*>(out), wbase,
                                             (long long)p.ws.nj * p.ws.S * p.ws.W);
                } else if (mode == 2) {
                    if (have_acc)
                        epilogue_mtile<2, float>(ta, nc, true, vrow, nl, K, static_cast<float*>(out), rowbase,
                                                 kstride);
                } else if constexpr (SPEC == 0) {
                    if (out_dtype == 2) {
                        epilogue_mtile<1, float>(ta, nc, have_acc, vrow, nl, K, static_cast<float*>(out), rowbase,
                                                 kstride);
                    } else if (out_dtype == 0) {
                        epilogue_mtile<1, __nv_bfloat16>(ta, nc, have_acc, vrow, nl, K,
                                                         static_cast<__nv_bfloat16*>(out), rowbase, kstride);
                    } else {
                        epilogue_mtile<1, __half>(ta, nc, have_acc, vrow, nl, K, static_cast<__half*>(out),
                                                  rowbase, kstride);
                    }
                }
            }
        }
    }
    if (p.staged) {
        // Write the CTA's dW block, Gm*K*T*C elements in dW order, four
        // consecutive channels at a time: element (g0 + gl, k, tap, c) is row
        // (atom % 2) * 64 + cw % 64 of M-tile atom / 2, cw = gl * C + c, and
        // column (x-block) * 64 + gl * K + k (gl * K + k without x-blocks) of the
        // dump.  Vector fp32 atomic adds (atomic) or stores into the split's
        // workspace rows (deterministic; a row of T*C elements, a multiple of 4,
        // never splits a vector across slices).
        named_bar_sync(3, kIgThreads);
        const float* dump = reinterpret_cast<const float*>(smem);
        const int C = p.C, K = p.K, T = p.T, TC = T * C, C4 = C >> 2, xs = p.xs, X = xs ? xs : 1;
        const int nv4 = p.Gm * K * TC / 4;
        const long long e0 = (long long)g0 * K * TC;
        for (int i = threadIdx.x; i < nv4; i += kIgThreads) {
            int rest = i / C4;
            const int c = (i - rest * C4) * 4;
            const int tap = rest % T;
            rest /= T;
            const int k = rest % K, gl = rest / K;
            const int x = tap % X;
            const int cw = gl * C + c, cc = cw >> 6;
            const int a = p.atom_of[(tap / X) * p.ncc + cc];
            const int rowi = (a & 1) * 64 + (cw & 63);
            const int col = (xs ? (xs - 1 - x) * 64 : 0) + gl * K + k;
            const float4 v = *reinterpret_cast<const float4*>(dump + ((a >> 1) * p.Nmma + col) * 128 + rowi);
            const long long e = e0 + 4LL * i;
            if (p.mode == 2) {
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(static_cast<float*>(p.out) + e),
                             "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                             : "memory");
            } else {
                const long long r = (long long)(g0 + gl) * K + k;
                const int xe = tap * C + c;
                const int j = xe / p.ws.W;
                float* o = static_cast<float*>(p.out) +
                           ((r * p.ws.nj + j) * p.ws.S + split) * (long long)p.ws.W + (xe - j * p.ws.W);
                *reinterpret_cast<float4*>(o) = v;
            }
        }
    }
    if (p.clq > 1) {
        cluster_sync_all();  // every CTA of the cluster has staged its partial sums
        cluster_reduce_store(p, smem_u32(smem), mtn, atom0, c_al, g0, k_base, p.out, split / p.clq, warp, lane);
        cluster_sync_all();  // no CTA leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, (uint32_t)p.tmem_cols);
    }
}

// dW = 0 before atomic split-K accumulation (the page's Preprocess zeroes the
// output when k_batch > 1).  Launched just before the main kernel, which is a
// programmatic dependent of it: the main kernel's CTAs start at once and wait
// for this grid (griddepcontrol.wait) only before their first atomic add.
__global__ void __launch_bounds__(256) zero_f32_kernel(float* __restrict__ p, long long n)
{
    // It is itself a programmatic dependent of the kernel before it on the
    // stream: it waits for that kernel before letting the main kernel launch,
    // so the main kernel may read X and dY without waiting.
    pdl_wait();
    pdl_launch_dependents();
    const long long n4 = n >> 2;
    const long long stride = (long long)gridDim.x * blockDim.x;
    float4* p4 = reinterpret_cast<float4*>(p);  // 16-byte aligned (checked on the host)
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
        p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0.f;
}

// dW = cast(ws) after atomic accumulation of a 16-bit dW into the fp32
// workspace ws (round to nearest even).  A programmatic dependent of the main
// kernel: it may start at once and waits for that grid before reading.
template <typename OUT>
__global__ void __launch_bounds__(256) cast_f32_kernel(const float* __restrict__ ws, OUT* __restrict__ dw, long long n)
{
    pdl_launch_dependents();
    pdl_wait();
    const long long n4 = n >> 2;
    const long long stride = (long long)gridDim.x * blockDim.x;
    const float4* w4 = reinterpret_cast<const float4*>(ws);  // 16-byte aligned (checked on the host)
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = w4[i];
        unsigned short b[4];
        if constexpr (std::is_same<OUT, __nv_bfloat16>::value) {
            b[0] = __bfloat16_as_ushort(__float2bfloat16_rn(v.x)), b[1] = __bfloat16_as_ushort(__float2bfloat16_rn(v.y));
            b[2] = __bfloat16_as_ushort(__float2bfloat16_rn(v.z)), b[3] = __bfloat16_as_ushort(__float2bfloat16_rn(v.w));
        } else {
            b[0] = __half_as_ushort(__float2half_rn(v.x)), b[1] = __half_as_ushort(__float2half_rn(v.y));
            b[2] = __half_as_ushort(__float2half_rn(v.z)), b[3] = __half_as_ushort(__float2half_rn(v.w));
        }
        // Four 16-bit values as one 8-byte store (dW is 16-byte aligned).
        const uint2 packed = make_uint2((unsigned)b[0] | ((unsigned)b[1] << 16), (unsigned)b[2] | ((unsigned)b[3] << 16));
        *reinterpret_cast<uint2*>(dw + 4 * i) = packed;
    }
    for (long long i = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        if constexpr (std::is_same<OUT, __nv_bfloat16>::value)
            dw[i] = __float2bfloat16_rn(ws[i]);
        else
            dw[i] = __float2half_rn(ws[i]);
    }
}

// Stage 2 of the deterministic split-K mode (the two-stage wgrad that PR
// #11602 and PR #12359 refer to): dW = cast(sum over splits of ws[s]) in a
// fixed order that depends on S only: for S >= 8 the splits fall into four
// contiguous ranges, each summed in index order, and the four range sums are
// added in range order; for S < 8 one range.  The result is bitwise
// reproducible.
__device__ __forceinline__ void store_cast(void* dw, long long i, float a, int out_dtype)
{
    if (out_dtype == 2)
        static_cast<float*>(dw)[i] = a;
    else if (out_dtype == 0)
        static_cast<__nv_bfloat16*>(dw)[i] = __float2bfloat16_rn(a);
    else
        static_cast<__half*>(dw)[i] = __float2half_rn(a);
}

constexpr int kRedThreads = 256;
constexpr int kRedGroups = 4;
constexpr uint32_t kRedPiece = 16384;  // bytes per bulk copy

__host__ __device__ __forceinline__ int red_groups(int S) { return S >= 8 ? kRedGroups : 1; }
static_assert(kRedGroups == 4, "slices_reduce_store maps (slice, range) pairs with shifts by 2");

// Sum nsl consecutive slices staged in shared memory -- slice sl0 + k at
// sm + k * S * W, with kRedGroups * W floats of scratch at part + k * kRedGroups * W
// -- in the fixed order and store their elements of dW.  Every thread of the CTA
// calls it (it synchronises them once).  W <= 128 (the planner's slice width),
// so a slice row is at most 32 float4 columns: pass 1 gives each warp one
// (slice, split range) and each lane one float4 column; pass 2 gives each
// thread one element.  The index arithmetic is shifts and one 32-bit division
// per element: with general divisions per item (and a 64-bit one per element)
// the two passes took ~2,300 cycles on the 56x56 workload's slices, against
// the few hundred their loads and adds need.
__device__ __forceinline__ void slices_reduce_store(const float* sm, float* part, const WsLayout& w, long long sl0,
                                                    int nsl, void* dw, int out_dtype)
{
    const int S = w.S, W = w.W;
    const int G = red_groups(S);  // 1 or kRedGroups (= 4)
    const int W4 = W >> 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    // Pass 1: range g of slice k is summed in index order, four independent
    // float4 chains per lane (16-byte shared-memory loads).
    for (int t = warp; t < nsl * G; t += nwarps) {
        const int k = G == 1 ? t : t >> 2;
        const int g = t - k * G;
        const int s0 = G == 1 ? 0 : (S * g) >> 2, s1 = G == 1 ? S : (S * (g + 1)) >> 2;
        if (lane < W4) {
            const float4* q = reinterpret_cast<const float4*>(sm + ((size_t)k * S + s0) * W) + lane;
            float4 a = q[0];
            q += W4;
            int s = s0 + 1;
            for (; s + 4 <= s1; s += 4, q += 4 * W4) {
                float4 v[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) v[jj] = q[jj * W4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) a.x += v[jj].x, a.y += v[jj].y, a.z += v[jj].z, a.w += v[jj].w;
            }
            for (; s < s1; ++s, q += W4) a.x += q[0].x, a.y += q[0].y, a.z += q[0].z, a.w += q[0].w;
            reinterpret_cast<float4*>(part + ((size_t)k * kRedGroups + g) * W)[lane] = a;
        }
    }
    __syncthreads();
    // Pass 2: the range sums of each element added in range order.
    for (int t = threadIdx.x; t < nsl * 128; t += blockDim.x) {
        const int k = t >> 7, i = t & 127;
        if (i >= W) continue;
        const int sl = (int)(sl0 + k);  // slice indices fit 31 bits (checked on the host)
        const int r = sl / w.nj;
        const int x0 = (sl - r * w.nj) * W;
        if (x0 + i >= w.L) continue;  // past the end of the row (its last slice)
        const float* pk = part + (size_t)k * kRedGroups * W;
        float a = pk[i];
        for (int g = 1; g < G; ++g) a += pk[g * W + i];
        store_cast(dw, (long long)r * w.L + x0 + i, a, out_dtype);
    }
}

// Bulk path: CTA b owns workspace slices [b * spc, (b + 1) * spc) (spc > 1 when
// slices are small: W elements of one dW row each), whose S partials are one
// contiguous block; one warp pulls it into shared memory with a few large
// cp.async.bulk copies, then the threads add the split ranges.  Launched with
// programmatic dependent launch: its set-up overlaps the split-K kernel's
// tail, and it waits for that kernel's writes with griddepcontrol.wait.
__global__ void __launch_bounds__(kRedThreads)
    reduce_splits_bulk_kernel(const float* __restrict__ ws, void* __restrict__ dw, const WsLayout w, int out_dtype,
                              int spc, long long n_slices)
{
    extern __shared__ uint8_t red_raw[];
    float* sm = align_shared<float>(red_raw, 128);
    __shared__ uint64_t bar;
    pdl_launch_dependents();  // the next call's first kernel waits for this grid before it reads
    const long long sl0 = (long long)blockIdx.x * spc;
    const int nsl = (int)min((long long)spc, n_slices - sl0);
    const uint32_t total = (uint32_t)nsl * (uint32_t)w.S * (uint32_t)w.W * 4u;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar, total);
    }
    __syncthreads();
    // Everything above may run while the split-K kernel is still finishing.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x < 32) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(ws + sl0 * w.S * w.W);
        for (uint32_t off = threadIdx.x * kRedPiece; off < total; off += 32 * kRedPiece) {
            const uint32_t size = min(kRedPiece, total - off);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(sm) + off),
                "l"(src + off), "r"(size), "r"(smem_u32(&bar))
                : "memory");
        }
    }
    if (!__syncthreads_and(mbar_wait(&bar, 0))) return;  // one decision for the whole CTA
    slices_reduce_store(sm, sm + (size_t)spc * w.S * w.W, w, sl0, nsl, dw, out_dtype);
}

// Register path: one CTA per workspace slice (W <= 128 elements), warp g adds
// split range g (the ranges of red_groups) of the slice's float4 columns, lane =
// column, with every load of its range issued before the first add (the loads
// come from L2, where the split-K kernel has just written them, so one round
// trip covers them all); then each element's range sums are added in range
// order.  The same order as the bulk path, bit for bit.
constexpr int kRegMaxRange = 32;  // splits one lane holds at once (larger ranges loop)
__global__ void __launch_bounds__(128)
    reduce_splits_regs_kernel(const float* __restrict__ ws, void* __restrict__ dw, const WsLayout w, int out_dtype)
{
    __shared__ float4 part[kRedGroups][32];
    pdl_launch_dependents();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int S = w.S, W = w.W, W4 = W >> 2, G = red_groups(S);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long sl = blockIdx.x;
    if (warp < G && lane < W4) {
        const int s0 = G == 1 ? 0 : (S * warp) >> 2, s1 = G == 1 ? S : (S * (warp + 1)) >> 2;
        const float4* q = reinterpret_cast<const float4*>(ws + (sl * S + s0) * (long long)W) + lane;
        float4 a = __ldcg(q);
        int s = s0 + 1;
        q += W4;
        while (s < s1) {
            const int n = min(kRegMaxRange, s1 - s);
            float4 v[kRegMaxRange];
#pragma unroll
            for (int j = 0; j < kRegMaxRange; ++j)
                if (j < n) v[j] = __ldcg(q + j * W4);
#pragma unroll
            for (int j = 0; j < kRegMaxRange; ++j)
                if (j < n) a.x += v[j].x, a.y += v[j].y, a.z += v[j].z, a.w += v[j].w;
            s += n;
            q += n * W4;
        }
        part[warp][lane] = a;
    }
    __syncthreads();
    const int i = threadIdx.x;
    if (i >= W) return;
    const int r = (int)(sl / w.nj);
    const int x0 = (int)(sl - (long long)r * w.nj) * W;
    if (x0 + i >= w.L) return;
    const float* p0 = reinterpret_cast<const float*>(&part[0][0]);
    float a = p0[i];
    for (int g = 1; g < G; ++g) a += p0[g * 128 + i];
    store_cast(dw, (long long)r * w.L + x0 + i, a, out_dtype);
}

// Fallback for split counts whose slice block does not fit shared memory: one
// thread per element, same layout and summation order.
__global__ void __launch_bounds__(kRedThreads)
    reduce_splits_kernel(const float* __restrict__ ws, void* __restrict__ dw, long long E, const WsLayout w,
                         int out_dtype)
{
    pdl_launch_dependents();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long i = (long long)blockIdx.x * kRedThreads + threadIdx.x;
    if (i >= E) return;
    const int S = w.S, G = red_groups(S);
    const long long o0 = ws_offset(w, i, 0);
    float a = 0.f;
    for (int g = 0; g < G; ++g) {
        const int s0 = S * g / G, s1 = S * (g + 1) / G;
        float q = ws[o0 + (long long)s0 * w.W];
        for (int s = s0 + 1; s < s1; ++s) q += ws[o0 + (long long)s * w.W];
        a = g == 0 ? q : a + q;
    }
    store_cast(dw, i, a, out_dtype);
}

}  // namespace wg
