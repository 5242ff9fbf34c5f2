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
// Warp roles (192 threads): warp 0 lane 0 issues TMA; warp 1 owns TMEM and its
// lane 0 issues tcgen05.mma; warps 2..5 read TMEM (lane quadrant = warp % 4)
// and store dW / atomically add / write the split-K workspace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"

namespace wg {

// Most M-tiles one CTA accumulates (TMEM columns = M-tiles x Nt <= 512).
constexpr int kMaxMt = 16;

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
    int patch[3];
    int patch_bytes, patch_tx;
    int n_patches, dy_off, slot_bytes, stage_bytes, stages;
    int tmem_cols;
    uint32_t idesc;
    int mode;       // 1 direct, 2 atomic, 3 workspace
    int out_dtype;  // wg_dtype
    int clq;        // CTAs per cluster along the split (1: no cluster reduction)
    void* out;
    long long split_stride;  // elements between the workspace slices of consecutive clusters
    unsigned char patch_ph[32][4];
    unsigned int atom_off[256];
    unsigned short atom_tap[256];
    unsigned char atom_cc[256];
    // K-step part of the A descriptor, the same for every K-tile: row offset of
    // the step's first 8-pixel group (start-address field) and the byte offset
    // of its second group (SBO field).  Filled on the host.
    unsigned long long kd_table[16];
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Epilogue of one M-tile for one warp: TMEM -> registers -> global, in chunks
// of 16 columns.  MODE 1 stores dW in OUT (fp32, bf16 or fp16), MODE 2 adds
// to fp32 dW with global atomics, MODE 3 stores fp32 to the split's workspace
// slice.  Each lane owns one row (tap, c); k runs over the chunk's columns.
template <int MODE, typename OUT>
__device__ __forceinline__ void epilogue_mtile(uint32_t taddr, int ncols, bool have_acc, bool vrow, int n_lo, int K,
                                               OUT* __restrict__ out, long long rowbase, long long kstride)
{
    for (int c16 = 0; c16 < ncols; c16 += 16) {
        float v[16];
        if (have_acc) {
            tmem_ld16(taddr + (uint32_t)c16, v);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
        }
        if (!vrow) continue;
        const int k0 = c16 - n_lo;
        OUT* o = out + rowbase + (long long)k0 * kstride;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int k = k0 + j;
            if (k >= 0 && k < K) {
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

__device__ __forceinline__ void store_elem(int mode, int out_dtype, void* out, long long i, float v)
{
    if (mode == 2) {
        red_add_f32(static_cast<float*>(out) + i, v);
    } else if (mode == 3 || out_dtype == 2) {
        static_cast<float*>(out)[i] = v;
    } else if (out_dtype == 0) {
        static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half*>(out)[i] = __float2half_rn(v);
    }
}

// Cluster reduction of the split-K partial sums, run by the four epilogue
// warps of every CTA of a cluster once each CTA has staged its accumulators in
// its own shared memory, column-major (red[(m * Nt + col) * 128 + row]).  The
// mtn * Nt columns are dealt out to the cluster's CTAs in contiguous ranges;
// for each of its columns a warp reads the 128 rows (lane = rows lane,
// lane + 32, lane + 64, lane + 96) from every CTA of the cluster through
// distributed shared memory, adds them in rank order -- a fixed order, so the
// result is reproducible -- and stores the sums (the dW values, or the
// cluster's partial sums) as whole 128-byte rows of consecutive channels.
__device__ __forceinline__ void cluster_reduce_store(const IgParams& p, uint32_t red_s, int mtn, int atom0, int c_al,
                                                     int g0, int k_base, void* out, int ew, int lane)
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
    for (int u = u0 + ew; u < u1; u += 4) {
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
            if (rm[i].base >= 0 && k >= 0 && k < K) store_elem(mode, out_dtype, out, rm[i].base + k * kstride, a);
        }
    }
}

struct MmaArgs {
    uint64_t b0;        // dY descriptor of stage 0, K-step 0
    uint32_t idesc, Nt, stage16;
    int ksteps, stages;
};

// The MMA issuer, run by a whole converged warp; one elected lane issues a
// K-step's MT MMAs.  Every operand is a sum of 64-bit parts whose fields never
// overlap: the M-tile part ab[m] (start of its first atom in stage 0, LBO to
// its second atom), the K-step part kdt[ks] (from the kernel parameters) and
// the stage offset.  The K-step loop is unrolled against the parameter table:
// descriptor operands built from runtime geometry inside the loop halved the
// MMA issue rate.
template <int MT>
__device__ __forceinline__ void mma_mainloop(const MmaArgs a, const uint64_t (&ab)[kMaxMt], uint64_t* full,
                                             uint64_t* empty, uint64_t* accb, uint32_t tbase, int nk,
                                             const unsigned long long* __restrict__ kdt)
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
            const uint64_t bdesc = b0 + soff + (uint64_t)(ks * 128);
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

__global__ void __launch_bounds__(192, 1)
    igemm_wgrad_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                       const __grid_constant__ IgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // [stages x stage_bytes][1 KB slack read by padding atoms][tail: barriers + tables]
    uint8_t* tail = smem + p.stages * p.stage_bytes + 1024;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);
    uint64_t* empty = full + 8;
    uint64_t* accb = empty + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);

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

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accb, 1);
        fence_mbar_init();
    }
    __syncthreads();  // barriers initialised: the producer may start
    if (warp == 1) {
        tmem_alloc(tslot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    // The TMEM address is read after the allocation, which the MMA and epilogue
    // warps wait for below; the producer does not need it.
    uint32_t tbase = 0;
    if (warp != 0) {
        named_bar_sync(1, 160);  // warps 1..5
        tc_fence_after();
        tbase = *tslot;
    }
#define MMA_ARGS ma, ab, full, empty, accb, tbase, nk, p.kd_table

    if (warp == 0) {
        if (lane == 0 && nk > 0) {
            // ------------------------------------------------ TMA producer
            tma_prefetch_desc(&tmx);
            tma_prefetch_desc(&tmy);
            const uint32_t tx = (uint32_t)(p.n_patches * p.patch_tx + p.n_katoms * p.slot_bytes);
            for (int i = 0; i < nk; ++i) {
                const int st = i % p.stages;
                const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
                if (i >= p.stages && !mbar_wait(&empty[st], ph ^ 1u)) break;
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
                    tma_load_5d(sb + p.dy_off + j * p.slot_bytes, &tmy, &full[st], k_base + 64 * j, wo0, ho0, do0, n0);
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
            ma.b0 = make_sdesc(sbase + (uint32_t)p.dy_off, (uint32_t)p.slot_bytes, 1024u, 2u, 0u);
            ma.idesc = p.idesc, ma.Nt = (uint32_t)Nt, ma.stage16 = (uint32_t)stage_bytes >> 4;
            ma.ksteps = ksteps, ma.stages = stages;
            switch (mtn) {
                case 1: mma_mainloop<1>(MMA_ARGS); break;
                case 2: mma_mainloop<2>(MMA_ARGS); break;
                case 3: mma_mainloop<3>(MMA_ARGS); break;
                case 4: mma_mainloop<4>(MMA_ARGS); break;
                case 5: mma_mainloop<5>(MMA_ARGS); break;
                case 6: mma_mainloop<6>(MMA_ARGS); break;
                case 7: mma_mainloop<7>(MMA_ARGS); break;
                case 8: mma_mainloop<8>(MMA_ARGS); break;
                case 9: mma_mainloop<9>(MMA_ARGS); break;
                case 10: mma_mainloop<10>(MMA_ARGS); break;
                case 11: mma_mainloop<11>(MMA_ARGS); break;
                case 12: mma_mainloop<12>(MMA_ARGS); break;
                case 13: mma_mainloop<13>(MMA_ARGS); break;
                case 14: mma_mainloop<14>(MMA_ARGS); break;
                case 15: mma_mainloop<15>(MMA_ARGS); break;
                default: mma_mainloop<16>(MMA_ARGS); break;
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        if (nk > 0) {
            mbar_wait_sleep(accb, 0);
            tc_fence_after();
        }
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int K = p.K, C = p.C, T = p.T, GC = p.GC, Gm = p.Gm, n_atoms = p.n_atoms, ncc = p.ncc, mode = p.mode;
        const int out_dtype = p.out_dtype;
        void* const out = p.out;
        const long long split_off = (long long)(split / p.clq) * p.split_stride;
        const uint32_t trow = tbase + ((uint32_t)(q * 32) << 16);
        const bool have_acc = nk > 0;
        if (p.clq > 1) {
            // Stage the accumulators for the cluster reduction in the (now idle)
            // pipeline buffers, column-major so that a warp's stores are
            // consecutive words.
            float* red = reinterpret_cast<float*>(smem);
            for (int m = 0; m < mtn; ++m)
                for (int c16 = 0; c16 < Nt; c16 += 16) {
                    float v[16];
                    if (have_acc) {
                        tmem_ld16(trow + (uint32_t)(m * Nt + c16), v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) red[(m * Nt + c16 + j) * 128 + row] = v[j];
                }
        }
        for (int m = 0; m < mtn && p.clq == 1; ++m) {
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
            const long long rowbase = ((long long)gr * K * T + tap) * C + c;
            const long long kstride = (long long)T * C;
            const uint32_t ta = trow + (uint32_t)(m * Nt);
            if (mode == 3) {
                epilogue_mtile<3, float>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<float*>(out) + split_off, rowbase,
                                         kstride);
            } else if (mode == 2) {
                if (have_acc)
                    epilogue_mtile<2, float>(ta, Nt, true, vrow, n_lo, K, static_cast<float*>(out), rowbase, kstride);
            } else if (out_dtype == 2) {
                epilogue_mtile<1, float>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<float*>(out), rowbase, kstride);
            } else if (out_dtype == 0) {
                epilogue_mtile<1, __nv_bfloat16>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<__nv_bfloat16*>(out),
                                                 rowbase, kstride);
            } else {
                epilogue_mtile<1, __half>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<__half*>(out), rowbase, kstride);
            }
        }
    }
    if (p.clq > 1) {
        cluster_sync_all();  // every CTA of the cluster has staged its partial sums
        if (warp >= 2) {
            void* out = p.mode == 3 ? (void*)(static_cast<float*>(p.out) + (long long)(split / p.clq) * p.split_stride)
                                    : p.out;
            cluster_reduce_store(p, smem_u32(smem), mtn, atom0, c_al, g0, k_base, out, warp - 2, lane);
        }
        cluster_sync_all();  // no CTA leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, (uint32_t)p.tmem_cols);
    }
}

// Stage 2 of the deterministic split-K mode (the two-stage wgrad that PR
// #11602 and PR #12359 refer to): dW = cast(sum over splits of ws[s]), each
// element summed over s = 0, 1, ..., S-1 in that order, so the result is
// bitwise reproducible.
//
// Bulk path (dW element count a multiple of 4): CTA b owns `chunk` consecutive
// elements; one thread copies that slice of every split into shared memory
// with cp.async.bulk (all S copies in flight at once), then each thread sums
// its elements from shared memory.  Launched with programmatic dependent
// launch: it waits for the split-K kernel's writes with griddepcontrol.wait.
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

__global__ void __launch_bounds__(kRedThreads)
    reduce_splits_bulk_kernel(const float* __restrict__ ws, void* __restrict__ dw, long long E, int S, int out_dtype,
                              int chunk)
{
    extern __shared__ uint8_t red_raw[];
    float* sm = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(red_raw) + 127) & ~uintptr_t(127));
    __shared__ uint64_t bar;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long e0 = (long long)blockIdx.x * chunk;
    const int n = (int)min((long long)chunk, E - e0);
    const uint32_t nbytes = (uint32_t)n * 4u;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar, nbytes * (uint32_t)S);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        // The copies are issued by a whole warp, one split per lane at a time.
        for (int s = threadIdx.x; s < S; s += 32) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(sm + (size_t)s * chunk)),
                "l"(ws + (long long)s * E + e0), "r"(nbytes), "r"(smem_u32(&bar))
                : "memory");
        }
    }
    if (!mbar_wait(&bar, 0)) return;
    for (int i = threadIdx.x; i < n; i += kRedThreads) {
        const float* col = sm + i;
        float a = col[0];
#pragma unroll 8
        for (int s = 1; s < S; ++s) a += col[(size_t)s * chunk];
        store_cast(dw, e0 + i, a, out_dtype);
    }
}

// Fallback for element counts that are not a multiple of 4: one thread per
// element, same summation order.
__global__ void __launch_bounds__(kRedThreads)
    reduce_splits_kernel(const float* __restrict__ ws, void* __restrict__ dw, long long E, int S, int out_dtype)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long i = (long long)blockIdx.x * kRedThreads + threadIdx.x;
    if (i >= E) return;
    float a = ws[i];
    for (int s = 1; s < S; ++s) a += ws[(long long)s * E + i];
    store_cast(dw, i, a, out_dtype);
}

}  // namespace wg
