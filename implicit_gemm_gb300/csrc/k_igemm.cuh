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

#include "ptx.cuh"

namespace wg {

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
    void* out;
    long long split_stride;
    unsigned char patch_ph[32][4];
    unsigned int atom_off[256];
    unsigned short atom_tap[256];
    unsigned char atom_cc[256];
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

__device__ __forceinline__ void store_out(const IgParams& p, long long idx, int split, float v)
{
    if (p.mode == 2) {
        red_add_f32(static_cast<float*>(p.out) + idx, v);
    } else if (p.mode == 3) {
        static_cast<float*>(p.out)[split * p.split_stride + idx] = v;
    } else if (p.out_dtype == 2) {
        static_cast<float*>(p.out)[idx] = v;
    } else if (p.out_dtype == 0) {
        static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half*>(p.out)[idx] = __float2half_rn(v);
    }
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
    uint32_t* s_aoff = tslot + 4;     // [32] stage offset of an M-tile's first atom
    uint32_t* s_lbo = s_aoff + 32;    // [32] offset from the first to the second atom
    uint32_t* s_krow = s_lbo + 32;    // [16] patch-row byte offset of a K-step's first 8-pixel group
    uint32_t* s_ksbo = s_krow + 16;   // [16] byte offset of its second group

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
        for (int m = 0; m < mtn; ++m) {
            const int a = atom0 + 2 * m;
            uint32_t off_a, off_b;
            if (p.halo) {
                off_a = p.atom_off[a];
                off_b = (a + 1 < p.n_atoms) ? p.atom_off[a + 1] : off_a + 1024;
            } else {
                off_a = (uint32_t)(2 * m) * p.patch_bytes;
                off_b = off_a + p.patch_bytes;
            }
            s_aoff[m] = off_a;
            s_lbo[m] = off_b - off_a;
        }
        const int PW = p.patch[0], PH = p.patch[1], PD = p.patch[2];
        for (int ks = 0; ks < p.ksteps; ++ks) {
            uint32_t prow[2];
            for (int h = 0; h < 2; ++h) {
                int r = 16 * ks + 8 * h;
                const int iw = r % p.box[0];
                r /= p.box[0];
                const int ih = r % p.box[1];
                r /= p.box[1];
                const int id = r % p.box[2];
                const int in = r / p.box[2];
                prow[h] = (uint32_t)(((in * PD + id) * PH + ih) * PW + iw);
            }
            s_krow[ks] = prow[0] * 128u;
            s_ksbo[ks] = (prow[1] - prow[0]) * 128u;
        }
    }
    if (warp == 1) {
        tmem_alloc(tslot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

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
        if (lane == 0 && nk > 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t sbase = smem_u32(smem);
            for (int i = 0; i < nk; ++i) {
                const int st = i % p.stages;
                const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
                if (!mbar_wait(&full[st], ph)) break;
                tc_fence_after();
                const uint32_t stb = sbase + (uint32_t)(st * p.stage_bytes);
                for (int ks = 0; ks < p.ksteps; ++ks) {
                    const uint64_t bdesc =
                        make_sdesc(stb + (uint32_t)p.dy_off + (uint32_t)ks * 2048u, (uint32_t)p.slot_bytes, 1024u, 2u, 0u);
                    const uint32_t krow = s_krow[ks], ksbo = s_ksbo[ks];
                    for (int m = 0; m < mtn; ++m) {
                        const uint64_t adesc = make_sdesc(stb + s_aoff[m] + krow, s_lbo[m], ksbo, 2u, 0u);
                        umma_f16(tbase + (uint32_t)(m * p.Nt), adesc, bdesc, p.idesc, (i | ks) != 0 ? 1u : 0u);
                    }
                }
                umma_commit(&empty[st]);
            }
            umma_commit(accb);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        if (nk > 0) {
            mbar_wait(accb, 0);
            tc_fence_after();
        }
        const int q = warp & 3;
        const int row = q * 32 + lane;
        for (int m = 0; m < mtn; ++m) {
            const int atom = atom0 + 2 * m + (row >> 6);
            bool vrow = atom < p.n_atoms;
            int tap = 0, cc = 0;
            if (vrow) {
                if (p.halo) {
                    tap = p.atom_tap[atom];
                    cc = p.atom_cc[atom];
                } else {
                    tap = atom / p.ncc;
                    cc = atom - tap * p.ncc;
                }
            }
            const int cg = c_al + cc * 64 + (row & 63);
            const int gr = cg / p.C;
            const int c = cg - gr * p.C;
            vrow = vrow && cg < p.GC && gr >= g0 && gr < g0 + p.Gm;
            const int n_lo = gr * p.K - k_base;
            const long long rowbase = ((long long)gr * p.K * p.T + tap) * p.C + c;
            const long long kstride = (long long)p.T * p.C;
            for (int c16 = 0; c16 < p.Nt / 16; ++c16) {
                float v[16];
                if (nk > 0) {
                    tmem_ld16(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * p.Nt + c16 * 16), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
                if (vrow && !(p.mode == 2 && nk == 0)) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int k = c16 * 16 + j - n_lo;
                        if (k >= 0 && k < p.K) store_out(p, rowbase + k * kstride, split, v[j]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, (uint32_t)p.tmem_cols);
    }
}

// Stage 2 of the deterministic split-K mode: dW = cast(sum over s = 0..S-1 of
// ws[s]), the splits summed in index order (reading of the two-stage wgrad of
// PR #10571 as referenced by PR #11602 and PR #12359).
__global__ void reduce_splits_kernel(const float* __restrict__ ws, void* __restrict__ dw, long long E, int S,
                                     int out_dtype)
{
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nth = (long long)gridDim.x * blockDim.x;
    if ((E & 3) == 0) {
        const long long E4 = E >> 2;
        const float4* w4 = reinterpret_cast<const float4*>(ws);
        for (long long i = tid; i < E4; i += nth) {
            float4 a = w4[i];
            for (int s = 1; s < S; ++s) {
                const float4 b = w4[(long long)s * E4 + i];
                a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
            }
            if (out_dtype == 2) {
                reinterpret_cast<float4*>(dw)[i] = a;
            } else if (out_dtype == 0) {
                __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(dw) + 2 * i;
                o[0] = __floats2bfloat162_rn(a.x, a.y);
                o[1] = __floats2bfloat162_rn(a.z, a.w);
            } else {
                __half2* o = reinterpret_cast<__half2*>(dw) + 2 * i;
                o[0] = __floats2half2_rn(a.x, a.y);
                o[1] = __floats2half2_rn(a.z, a.w);
            }
        }
    } else {
        for (long long i = tid; i < E; i += nth) {
            float a = ws[i];
            for (int s = 1; s < S; ++s) a += ws[(long long)s * E + i];
            if (out_dtype == 2)
                static_cast<float*>(dw)[i] = a;
            else if (out_dtype == 0)
                static_cast<__nv_bfloat16*>(dw)[i] = __float2bfloat16_rn(a);
            else
                static_cast<__half*>(dw)[i] = __float2half_rn(a);
        }
    }
}

}  // namespace wg
