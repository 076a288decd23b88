// Diagonal-tile factor of the blocked path on a thread-block cluster, for
// few matrices (sm_103a).
//
// One matrix's diagonal tile (order kb <= 128) is factored by a cluster of
// C blocks on C SMs (C = 8, or 16 where such a cluster fits) instead of one
// block on one SM.  On GB300 a warp issues
// at most one FP64 instruction every 64 cycles whatever its active lanes, so
// a 128-wide tile on one SM is bound by that SM's FP64 rate (about 1.7
// multiply-adds per cycle) and by the column chain; C SMs share the first.
//
// The tile's rows are dealt round-robin: block r of the cluster holds rows
// i = r, r + C, ... in shared memory.  The factor runs right-looking over
// 16-column panels (jaxmg docs "Cholesky factorization": the tiled potrf's
// diagonal factor, panel solve and trailing update, here within one tile),
// each panel in three steps separated by cluster barriers:
//   A. every block writes its rows' panel columns into every block's panel
//      buffer (distributed shared memory);
//   B. every block factors the panel's 16 x 16 diagonal block from its own
//      copy (the same arithmetic in every block, so the same result), four
//      warps sharing the column updates so the chain of reciprocal square
//      roots is not held up by them;
//   C. every block solves its own rows of the panel against that block and
//      hands the results to every block's panel buffer;
//   D. every block applies the panel to the trailing columns of its rows.
// On request the cluster then also inverts the factored tile (for the
// tensor-core panel solve), each block 16 of its columns.
// Panel buffers alternate between panels, so step A of one panel never
// overwrites what another block may still read in step D of the previous.
//
// The arithmetic is that of the single-block tile factor: pivot d, 1 / l_jj =
// rsqrt(d), l_jj = d * rsqrt(d), the first pivot that is not > 0 (zero,
// negative, NaN) is the status; the order of the sums differs, so results
// agree with the other paths to rounding.  Every barrier is a hardware
// cluster barrier: no block spins on a flag.
#include <cooperative_groups.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace chol {

namespace cg = cooperative_groups;

namespace {

constexpr int kClThreads = 256;
constexpr int kPW = 16;        // panel width
constexpr int kPP = kPW + 1;   // pitch of a panel-buffer row
constexpr int kTileMax = 128;  // largest tile order

template <int C>
struct ClLayout {
    static constexpr int R = kTileMax / C;  // rows per block
    static constexpr int AP = kTileMax;     // pitch of a held row
    // element offsets (in T) of the shared-memory regions
    static constexpr int a_off = 0;                          // R x AP held rows
    static constexpr int pb_off = a_off + R * AP;            // 2 x 128 x kPP panel buffers
    static constexpr int h_off = pb_off + 2 * kTileMax * kPP;  // kPW x kPP scaled diagonal block
    static constexpr int col_off = h_off + kPW * kPP;        // 2 x kPW column hand-off
    static constexpr int rinv_off = col_off + 2 * kPW;       // kPW reciprocals
    static constexpr int elems = rinv_off + kPW;
    // with the inverse: the whole factor's rows scaled by 1 / l_ii (packed
    // lower, strictly below the diagonal) and the reciprocals 1 / l_ii
    static constexpr int hs_off = elems;
    static constexpr int rd_off = hs_off + kTileMax * (kTileMax + 1) / 2;
    static constexpr int elems_inv = rd_off + kTileMax;
};

template <typename T, int C>
size_t cl_smem_bytes(bool with_inverse) {
    return (size_t)(with_inverse ? ClLayout<C>::elems_inv : ClLayout<C>::elems) * sizeof(T) + 16;
}

__device__ __forceinline__ int packed(int i, int j) { return i * (i + 1) / 2 + j; }

// 1 / sqrt(d) on the pivot chain.  float: rsqrtf.  double: a float seed
// (d's leading 24 bits as a float, by integer arithmetic; then rsqrtf, about
// 2^-22 relative error) and one step of Halley's iteration for the
// reciprocal square root in FP64, y1 = y0 (1 + e/2 + 3 e^2/8) with
// e = 1 - d y0^2, whose error is about (5/16) e^3 plus the rounding of its
// five FP64 operations: the chain's FP64 instructions (a warp issues one per
// 64 cycles here) are fewer than with rsqrt.  Pivots outside the float range,
// and those that are not positive or not finite (the status decides about
// them), take rsqrt.
__device__ __forceinline__ float pivot_rsqrt(float d) { return rsqrtf(d); }
__device__ __forceinline__ double pivot_rsqrt(double d) {
    const long long bits = __double_as_longlong(d);
    const int E = (int)((bits >> 52) & 0x7ff) - 1023;
    if (bits <= 0 || E < -125 || E > 125) return rsqrt(d);
    const float f = __int_as_float(((E + 127) << 23) | (int)((bits >> 29) & 0x7fffff));
    const int fb = __float_as_int(rsqrtf(f));
    const double y0 = __longlong_as_double(
        ((long long)(((fb >> 23) & 0xff) - 127 + 1023) << 52) | ((long long)(fb & 0x7fffff) << 29));
    const double h = d * y0;
    const double e = fma(-h, y0, 1.0);
    const double t = fma(0.375, e, 0.5);
    return fma(y0, e * t, y0);
}

// Rows of the held set at or below row `lo`: t = first .. cnt - 1.
template <int C>
__device__ __forceinline__ int first_at_or_below(int rank, int lo) {
    return lo <= rank ? 0 : (lo - rank + C - 1) / C;
}

template <typename T, int C>
__global__ void __launch_bounds__(kClThreads, 1)
cl_potrf_kernel(T* __restrict__ L, int32_t* __restrict__ status, int64_t batch, int n, int k0,
                int kb, T* __restrict__ Inv, int32_t* __restrict__ bal, int nt) {
    pdl_wait();
    using Lay = ClLayout<C>;
    constexpr int AP = Lay::AP;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* sm = reinterpret_cast<T*>(smem_raw);
    T* A = sm + Lay::a_off;
    T* PB = sm + Lay::pb_off;
    T* H = sm + Lay::h_off;
    T* colbuf = sm + Lay::col_off;
    T* rinv = sm + Lay::rinv_off;
    __shared__ int s_fail;
    __shared__ T s_piv[kPW];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // rows held by this block: i = rank + C t, t < nrows
    const int nrows = kb > rank ? (kb - rank + C - 1) / C : 0;

    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        // nobody still reads a panel buffer of the previous matrix
        cluster.sync();
        if (status != nullptr && status[b] != 0) continue;
        T* Lb = L + b * (int64_t)n * n;
        for (int e = tid; e < nrows * AP; e += kClThreads) {
            const int t = e / AP, j = e % AP, i = rank + C * t;
            A[t * AP + j] = (j <= i && j < kb) ? Lb[(int64_t)(k0 + i) * n + k0 + j] : T(0);
        }
        if (tid == 0) s_fail = INT_MAX;
        __syncthreads();
        bool failed = false;
        const int npanels = (kb + kPW - 1) / kPW;
        for (int q = 0; q < npanels; ++q) {
            const int c0 = q * kPW, w = min(kPW, kb - c0);
            T* pb = PB + (q & 1) * kTileMax * kPP;
            // A. this block's rows i >= c0, panel columns (zeros past w), to every block
            {
                const int t0 = first_at_or_below<C>(rank, c0);
                const int cnt = (nrows - t0) * kPW;
                for (int e = tid; e < cnt * C; e += kClThreads) {
                    const int d = e / cnt, f = e % cnt;
                    const int t = t0 + f / kPW, k = f % kPW, i = rank + C * t;
                    const T v = k < w ? A[t * AP + c0 + k] : T(0);
                    cluster.map_shared_rank(pb, d)[i * kPP + k] = v;
                }
            }
            cluster.sync();
            // B. the diagonal block (rows c0 .. c0 + 15 of pb), eight warps:
            // warp u holds columns u (lanes 0-15) and u + 8 (lanes 16-31), row
            // lane % 16, so that each column step costs every warp one FP64
            // instruction (a warp issues one per 64 cycles here) and the next
            // pivot's warp is never held up by updates of its other columns
            {
                const int r = lane & 15;
                const int col = warp + 8 * (lane >> 4);
                T a = pb[(c0 + r) * kPP + col];
                for (int j = 0; j < kPW; ++j) {
                    T* cb = colbuf + (j & 1) * kPW;
                    if (warp == (j & 7)) {
                        // (row j's own entry is d, so l_jj = d / sqrt(d) is the
                        // same product; the pivot's sign is checked after the
                        // loop, off the chain)
                        const T d = __shfl_sync(0xffffffffu, a, 16 * (j >> 3) + j);
                        const T ri = pivot_rsqrt(d);
                        if ((lane >> 4) == (j >> 3)) {
                            a *= ri;
                            cb[r] = a;
                        }
                        if (lane == 0) {
                            rinv[j] = j < w ? ri : T(0);
                            s_piv[j] = d;
                        }
                    }
                    __syncthreads();
                    if (col > j) a = fma(-cb[r], cb[col], a);
                }
                pb[(c0 + r) * kPP + col] = a;
                // the first pivot that is not > 0 (zero, negative, NaN); every
                // pivot was written before the last column's barrier
                if (warp == 0 && lane < w && !(s_piv[lane] > T(0))) atomicMin(&s_fail, lane);
            }
            __syncthreads();
            if (s_fail < w) {
                // the same pivot failed in every block of the cluster
                if (rank == 0 && tid == 0) status[b] = k0 + c0 + s_fail + 1;
                failed = true;
                break;
            }
            // the diagonal block's rows scaled by 1 / l_kk (strictly lower part)
            for (int e = tid; e < kPW * kPW; e += kClThreads) {
                const int k = e / kPW, m = e % kPW;
                H[k * kPP + m] = (m < k && k < w) ? pb[(c0 + k) * kPP + m] * rinv[k] : T(0);
            }
            // rows of this block inside the diagonal block: their factor rows
            {
                const int t0 = first_at_or_below<C>(rank, c0);
                for (int e = tid; e < (nrows - t0) * kPW; e += kClThreads) {
                    const int t = t0 + e / kPW, k = e % kPW, i = rank + C * t;
                    if (i < c0 + w && k <= i - c0) A[t * AP + c0 + k] = pb[i * kPP + k];
                }
            }
            __syncthreads();
            // C. this block's rows below the diagonal block: x = a L_D^-T, one
            // half-warp per row, lane k holding x_k
            {
                const int t0 = first_at_or_below<C>(rank, c0 + w);
                const int k = lane & 15;
                for (int t = t0 + 2 * warp + (lane >> 4); t - (lane >> 4) < nrows;
                     t += 2 * (kClThreads / 32)) {
                    const bool live = t < nrows;
                    const int i = rank + C * t;
                    T acc = live ? pb[i * kPP + k] * rinv[k] : T(0);
#pragma unroll
                    for (int m = 0; m < kPW - 1; ++m) {
                        const T xm = __shfl_sync(0xffffffffu, acc, m, 16);
                        if (k > m) acc = fma(-xm, H[k * kPP + m], acc);
                    }
                    if (live && k < w) {
                        A[t * AP + c0 + k] = acc;
#pragma unroll
                        for (int d = 0; d < C; ++d) cluster.map_shared_rank(pb, d)[i * kPP + k] = acc;
                    }
                }
            }
            cluster.sync();
            // D. trailing update of this block's rows: a_ij -= x_i . x_j for
            // c0 + w <= j <= i
            {
                const int lo = c0 + w;
                const int t0 = first_at_or_below<C>(rank, lo);
                // flattened (t, j) pairs; row t has i - lo + 1 of them
                int total = 0;
                for (int t = t0; t < nrows; ++t) total += rank + C * t - lo + 1;
                for (int e = tid; e < total; e += kClThreads) {
                    int t = t0, rem = e;
                    while (rem > rank + C * t - lo) {
                        rem -= rank + C * t - lo + 1;
                        ++t;
                    }
                    const int i = rank + C * t, j = lo + rem;
                    const T* xi = pb + i * kPP;
                    const T* xj = pb + j * kPP;
                    T acc = A[t * AP + j];
#pragma unroll
                    for (int k = 0; k < kPW; ++k) acc = fma(-xi[k], xj[k], acc);
                    A[t * AP + j] = acc;
                }
            }
            __syncthreads();
        }
        if (failed) continue;
        for (int e = tid; e < nrows * AP; e += kClThreads) {
            const int t = e / AP, j = e % AP, i = rank + C * t;
            if (j <= i) Lb[(int64_t)(k0 + i) * n + k0 + j] = A[t * AP + j];
        }
        if (Inv == nullptr) continue;
        // The inverse X = G^-1 of the factored tile G, written as a 128 x 128
        // matrix Inv[b] (zeros above the diagonal and beyond kb), for the
        // panel solve's product.  Every block receives the whole factor, its
        // rows scaled by 1 / g_ii (H_im = g_im / g_ii), then solves 16 of the
        // columns: G x = e_c by forward substitution in its right-looking
        // form, x_c = 1 / g_cc, then acc_i -= H_im x_m for the rows i > m,
        // x_m handed from the lane that owns row m by a shuffle.  Each block also
        // writes the balancing exponents ilogb(g_ii) of its own rows.
        T* Hs = sm + Lay::hs_off;
        T* rd = sm + Lay::rd_off;
        for (int e = tid; e < nrows * AP; e += kClThreads) {
            const int t = e / AP, j = e % AP, i = rank + C * t;
            if (j > i) continue;
            const T gii = A[t * AP + i];
            if (j == i) {
#pragma unroll 1
                for (int d = 0; d < C; ++d) cluster.map_shared_rank(rd, d)[i] = T(1) / gii;
                if (bal != nullptr)  // each block for its own rows
                    bal[b * (int64_t)nt * kTileMax + k0 + i] =
                        (gii > T(0) && isfinite(gii)) ? ilogb(gii) : 0;
            } else {
                const T h = A[t * AP + j] / gii;
#pragma unroll 1
                for (int d = 0; d < C; ++d) cluster.map_shared_rank(Hs, d)[packed(i, j)] = h;
            }
        }
        cluster.sync();
        T* Ib = Inv + b * (int64_t)kTileMax * kTileMax;
        constexpr int Q = kTileMax / 32;  // rows per lane
        for (int c = rank + C * warp; c < kTileMax; c += C * (kClThreads / 32)) {
            T acc[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) acc[q] = (lane + 32 * q == c && c < kb) ? rd[c] : T(0);
            for (int m = c; m < kb - 1; ++m) {
                const int slot = m >> 5;
                T v = acc[0];
#pragma unroll
                for (int q = 1; q < Q; ++q) v = slot == q ? acc[q] : v;
                const T xm = __shfl_sync(0xffffffffu, v, m & 31);
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    if (32 * q + 31 <= m) continue;  // (warp-uniform) no row of this slot is left
                    const int i = lane + 32 * q;
                    if (i > m && i < kb) acc[q] = fma(-Hs[packed(i, m)], xm, acc[q]);
                }
            }
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int i = lane + 32 * q;
                Ib[(int64_t)i * kTileMax + c] = (c < kb && i >= c && i < kb) ? acc[q] : T(0);
            }
        }
    }
    // no block leaves while another may still write into its shared memory
    cluster.sync();
}

// Launch with a cluster of C blocks (C = 16 is beyond the portable size of
// 8: the kernel is allowed it, and it is used only where the device can
// schedule such a cluster).
template <typename T, int C>
cudaError_t launch_cl_potrf(T* L, int32_t* status, int64_t batch, int n, int k0, int kb,
                            T* Inv, int32_t* bal, int nt, cudaStream_t stream) {
    auto kern = cl_potrf_kernel<T, C>;
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [&]() -> cudaError_t {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cl_smem_bytes<T, C>(true));
        if (r == cudaSuccess && C > 8)
            r = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return r;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, (unsigned)std::min<int64_t>(batch, 65535));
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = cl_smem_bytes<T, C>(Inv != nullptr);
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    // programmatic dependent launch (the kernel waits for its predecessor first)
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, L, status, batch, n, k0, kb, Inv, bal, nt);
}

// Whether a 16-block cluster of this kernel (with the inverse's shared
// memory) fits on the current device; checked once per device.
template <typename T>
bool cluster16_fits() {
    static PerDeviceInt fits;
    return fits.get([] {
        auto kern = cl_potrf_kernel<T, 16>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)cl_smem_bytes<T, 16>(true)) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess) {
            cudaGetLastError();
            return 1;  // 1: no (the cached value must be > 0)
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1);
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = cl_smem_bytes<T, 16>(true);
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 16;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 1;
        }
        return clusters >= 1 ? 2 : 1;  // 2: yes
    }) == 2;
}

}  // namespace

bool cluster_diag_pays(int64_t batch, int kb) {
    // one cluster of 8 or 16 SMs per matrix while the clusters leave most SMs idle
    return kb > 32 && kb <= kTileMax && batch * 8 <= device_sm_count();
}

template <typename T>
cudaError_t cluster_potrf_diag(T* L, int32_t* status, int64_t batch, int n, int k0, int kb,
                               T* Inv, int32_t* bal, cudaStream_t stream) {
    if (kb <= 0 || kb > kTileMax) return cudaErrorInvalidValue;
    const int nt = (n + kTileMax - 1) / kTileMax;
    // 16 SMs per matrix for one or a few matrices, where they fit
    if (batch * 16 <= device_sm_count() && cluster16_fits<T>())
        return launch_cl_potrf<T, 16>(L, status, batch, n, k0, kb, Inv, bal, nt, stream);
    return launch_cl_potrf<T, 8>(L, status, batch, n, k0, kb, Inv, bal, nt, stream);
}

template cudaError_t cluster_potrf_diag<float>(float*, int32_t*, int64_t, int, int, int, float*,
                                               int32_t*, cudaStream_t);
template cudaError_t cluster_potrf_diag<double>(double*, int32_t*, int64_t, int, int, int,
                                                double*, int32_t*, cudaStream_t);

}  // namespace chol
