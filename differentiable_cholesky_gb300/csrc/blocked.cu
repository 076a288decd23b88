// Blocked Cholesky forward and adjoint for n > 64 (square tiles of T = 32, 64
// or 128; the last tile of a row/column is ragged when T does not divide n).
//
// Forward: right-looking blocked potrf with L as the work buffer (A is only
// read, by the first kernel).  Per tile step k (jaxmg docs "Cholesky
// factorization", tile size T_A; the pages' own prior art is a distributed
// tiled factorisation, here the tiles stay on one GPU):
//   1. potrf_diag : factor the diagonal tile L_kk in shared memory (status on
//                   the first non-positive pivot, column k*T + j + 1);
//   2. trsm       : panel L_ik <- L_ik L_kk^-T for the rows below the tile;
//   3. gemm       : trailing update L_ij -= L_ik L_jk^T on the lower tiles.
// Only step 3 is a dense contraction.
//
// Adjoint: the symmetric-matrix derivative of Murray (2016) that NVIDIA/warp
// issue #1316's closing comment states as S = Phi(L^T adj_L) followed by two
// triangular solves, evaluated here by the same paper's blocked reverse sweep
// over a left-looking blocked factorisation (see blocked_adj): per tile column
// a triangular solve, three GEMM-shaped updates and a shared-memory reverse
// sweep of the diagonal tile, 2 n^3 / 3 flops in all instead of 7 n^3 / 3.
// Matrices whose status is non-zero are skipped by every kernel.
//
// The FP64 path is bound by the FP64 FMA pipe; every kernel keeps each SM's
// pipe fed with independent FMAs and does nothing else of consequence.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "chol_tile.cuh"
#include "kernels.h"

namespace chol {
namespace {

using chol_tile::cplx;
using chol_tile::detail::add;
using chol_tile::detail::conj;
using chol_tile::detail::madd;
using chol_tile::detail::re;
using chol_tile::detail::scale;
using chol_tile::detail::shfl_xor;
using chol_tile::detail::sub;

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// Lookahead of the float64 tensor-core forward: a second stream per device
// (and two events) on which the trailing update of step k, minus block column
// k + 1, runs beside step k + 1's diagonal factor and panel solve.  The
// caller's stream waits for it before it touches those columns again and
// before the forward returns, so the caller sees one stream's ordering.  The
// enqueue sequence of one forward holds the device's lock, so concurrent
// callers cannot interleave their event records.
// ---------------------------------------------------------------------------
struct SideStream {
    cudaStream_t s = nullptr;    // the updates beside the chain (default priority)
    cudaStream_t hi = nullptr;   // the chain itself (the device's highest priority)
    cudaEvent_t look = nullptr;  // the chain reached step k's lookahead column
    cudaEvent_t rest = nullptr;  // the side stream finished step k's remaining columns
    cudaEvent_t fork = nullptr;  // the caller's stream reached the forward / adjoint
    cudaEvent_t done = nullptr;  // the chain finished
};

SideStream g_side[kMaxDevices];
std::mutex g_side_lock[kMaxDevices];
std::atomic<uint64_t> g_side_made{0};

// The device's side streams (created on first use); false if there are none.
bool side_stream(int& dev, SideStream& out) {
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    const cudaError_t e = once_per_device(g_side_made, [&]() -> cudaError_t {
        SideStream sd;
        int least = 0, greatest = 0;
        cudaError_t r = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (r == cudaSuccess) r = cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking);
        if (r == cudaSuccess)
            r = cudaStreamCreateWithPriority(&sd.hi, cudaStreamNonBlocking, greatest);
        for (cudaEvent_t* ev : {&sd.look, &sd.rest, &sd.fork, &sd.done})
            if (r == cudaSuccess) r = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (r == cudaSuccess) g_side[dev] = sd;
        return r;
    });
    if (e != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    out = g_side[dev];
    return true;
}

// The chain of a lookahead call runs on the high-priority stream, so that
// when SMs free up the scheduler takes its (short, latency-bound) kernels
// before the side stream's bulk updates; it starts after the caller's stream
// has reached the call, and the caller's stream waits for the chain (which
// itself waits for the side stream's last work) before the call ends.
struct JoinSide {
    cudaStream_t main;   // the caller's stream
    cudaStream_t chain;  // where the chain runs: main, or the high-priority stream
    const SideStream* sd;
    bool pending = false;  // side work the chain has not waited for yet
    bool forked = false;   // chain != main
    cudaError_t start(bool look) {
        if (!look) return cudaSuccess;
        cudaError_t e = cudaEventRecord(sd->fork, main);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sd->hi, sd->fork, 0);
        if (e == cudaSuccess) {
            chain = sd->hi;
            forked = true;
        }
        return e;
    }
    cudaError_t finish() {
        cudaError_t e = cudaSuccess;
        if (pending) {
            e = cudaStreamWaitEvent(chain, sd->rest, 0);
            pending = false;
        }
        if (forked) {
            if (e == cudaSuccess) e = cudaEventRecord(sd->done, chain);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(main, sd->done, 0);
            forked = false;
        }
        return e;
    }
    ~JoinSide() { finish(); }
};

template <typename T> using real_t = typename chol_tile::detail::real_of<T>::type;

// Element-wise atomic add (a complex value adds its two parts separately).
__device__ __forceinline__ void atomic_add(float* p, float v) { atomicAdd(p, v); }
__device__ __forceinline__ void atomic_add(double* p, double v) { atomicAdd(p, v); }
template <typename R> __device__ __forceinline__ void atomic_add(cplx<R>* p, cplx<R> v) {
    atomicAdd(&p->re, v.re);
    atomicAdd(&p->im, v.im);
}

inline unsigned grid_y(int64_t batch) { return (unsigned)std::min<int64_t>(batch, 65535); }

__device__ __forceinline__ bool skip_matrix(const int32_t* status, int64_t b) {
    return status != nullptr && status[b] != 0;
}

// ---------------------------------------------------------------------------
// L = tril(A), status = 0
// ---------------------------------------------------------------------------
// A and L may be the same buffer (the in-place forward): each element is
// read and then written by the same thread.
template <typename T>
__global__ void __launch_bounds__(kThreads)
tril_copy_kernel(const T* A, T* L, int32_t* __restrict__ status, int64_t batch, int n) {
    const int64_t nn = (int64_t)n * n;
    const int64_t total = batch * nn;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = e % nn;
        const int i = (int)(w / n), j = (int)(w % n);
        L[e] = (j <= i) ? A[e] : T{};
    }
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < batch;
         b += (int64_t)gridDim.x * blockDim.x)
        status[b] = 0;
}

// ---------------------------------------------------------------------------
// Diagonal tile factor (one block per matrix), in shared memory.
// ---------------------------------------------------------------------------
template <typename T, int THREADS>
__global__ void __launch_bounds__(THREADS)
potrf_diag_kernel(T* __restrict__ L, int32_t* __restrict__ status, int64_t batch, int n,
                  int k0, int kb) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* S = reinterpret_cast<T*>(smem_raw);
    const int P = kb + 1;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (skip_matrix(status, b)) continue;
        T* Lb = L + b * (int64_t)n * n;
        __syncthreads();
        for (int e = threadIdx.x; e < kb * kb; e += blockDim.x) {
            const int r = e / kb, c = e % kb;
            S[r * P + c] = (c <= r) ? Lb[(int64_t)(k0 + r) * n + k0 + c] : T{};
        }
        __syncthreads();
        const int st = chol_tile::potrf<THREADS>(S, kb, chol_tile::RowMajor{P});
        if (st != 0) {
            if (threadIdx.x == 0) status[b] = k0 + st;
            continue;
        }
        for (int e = threadIdx.x; e < kb * kb; e += blockDim.x) {
            const int r = e / kb, c = e % kb;
            if (c <= r) Lb[(int64_t)(k0 + r) * n + k0 + c] = S[r * P + c];
        }
    }
}

// ---------------------------------------------------------------------------
// Triangular solves with a diagonal tile G of L, many right-hand sides.
// Each right-hand side ("vector") is solved by 4 consecutive lanes that split
// every dot product and combine it with two shuffles.
// ---------------------------------------------------------------------------
enum TrsmMode {
    TRSM_FWD_PANEL = 0,  // rows of L below tile k:        x L_kk^T = b  (G = L_kk, forward)
    TRSM_ADJ_M = 2       // rows of W below tile column J: m L_JJ = b    (G = L_JJ^T, backward)
};

constexpr int kVecPerBlock = kThreads / 4;

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads)
trsm_kernel(const T* L, T* W, const int32_t* __restrict__ status,
            int64_t batch, int n, int t0, int kb, int v_begin, int v_count) {
    using R = real_t<T>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int P = kb + 1;
    T* G = reinterpret_cast<T*>(smem_raw);          // kb x P
    T* V = G + (size_t)kb * P;                      // kVecPerBlock x P
    // kb reciprocals of G's (real) diagonal
    R* ginv = reinterpret_cast<R*>(V + (size_t)kVecPerBlock * P);
    const int vloc = threadIdx.x >> 2;
    const int q = threadIdx.x & 3;
    const int v0 = v_begin + blockIdx.x * kVecPerBlock;
    const int nv = min(kVecPerBlock, v_begin + v_count - v0);
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (skip_matrix(status, b)) continue;
        const T* Lb = L + b * (int64_t)n * n;
        T* Wb = W + b * (int64_t)n * n;
        __syncthreads();
        // G: lower tile (forward) or the transposed tile (backward)
        for (int e = threadIdx.x; e < kb * kb; e += blockDim.x) {
            const int r = e / kb, c = e % kb;  // coalesced over c in global memory
            const T x = (c <= r) ? Lb[(int64_t)(t0 + r) * n + t0 + c] : T{};
            if (MODE == TRSM_FWD_PANEL) G[r * P + c] = x;
            else G[c * P + r] = x;
        }
        // right-hand sides
        // vectors are rows v0.. of columns [t0, t0 + kb) (of L itself in the
        // forward panel, where W == L)
        for (int e = threadIdx.x; e < kb * kVecPerBlock; e += blockDim.x) {
            const int v = e / kb, m = e % kb;
            V[v * P + m] = (v < nv) ? Wb[(int64_t)(v0 + v) * n + t0 + m] : T{};
        }
        __syncthreads();
        for (int c = threadIdx.x; c < kb; c += blockDim.x) ginv[c] = rcp_t(re(G[c * P + c]));
        __syncthreads();
        {
            // every group runs the same sweep (idle groups on zero vectors
            // that are not stored), so the warp's shuffles stay convergent
            T* x = V + vloc * P;
            if (MODE == TRSM_FWD_PANEL) {
                for (int c = 0; c < kb; ++c) {
                    const T* g = G + c * P;
                    // x_c = (b_c - sum_{m<c} x_m conj(g_cm)) / g_cc
                    T s = T{};
                    for (int m = q; m < c; m += 4) s = madd(conj(g[m]), x[m], s);
                    s = add(s, shfl_xor(s, 1));
                    s = add(s, shfl_xor(s, 2));
                    if (q == 0) x[c] = scale(sub(x[c], s), ginv[c]);
                    __syncwarp();
                }
            } else {
                for (int c = kb - 1; c >= 0; --c) {
                    const T* g = G + c * P;
                    T s = T{};
                    for (int m = c + 1 + q; m < kb; m += 4) s = madd(g[m], x[m], s);
                    s = add(s, shfl_xor(s, 1));
                    s = add(s, shfl_xor(s, 2));
                    if (q == 0) x[c] = scale(sub(x[c], s), ginv[c]);
                    __syncwarp();
                }
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kb * kVecPerBlock; e += blockDim.x) {
            const int v = e / kb, m = e % kb;
            if (v < nv) Wb[(int64_t)(v0 + v) * n + t0 + m] = V[v * P + m];
        }
    }
}

// ---------------------------------------------------------------------------
// Tile GEMM: C_sub (BM x BM) = alpha * sum_kk opA(r, kk) opB(kk, c) + beta * C_sub
// over the tile schedules of the forward trailing update and the adjoint.
// ---------------------------------------------------------------------------
enum GemmMode {
    GEMM_FWD_TRAIL = 0,  // L_ij -= L_ik L_jk^T, k < j <= i
    // reverse sweep over tile column J = step (see blocked_adj):
    GEMM_REV_ROW = 4,    // W_JK -= Wbar_panel^T L_panel,K  (K <= J; split over the rows below)
    GEMM_REV_UPD = 5,    // W_IK -= W_IJ L_JK  (I > J, K < J)
    GEMM_REV_SYM = 6     // W_JK -= (W_JJ + W_JJ^T) L_JK  (K < J; W_JJ lower)
};

template <typename T>
struct GemmArgs {
    const T* A;   // operand matrices (batch-strided by n*n)
    const T* B;
    T* C;
    const int32_t* status;
    int64_t batch;
    int n;
    int tile;     // T
    int nt;       // tiles per side
    int step;     // k, I or J
    int kchunk;   // reduction length per blockIdx.z (split reduction)
    int atomic;   // 1: the epilogue adds with atomics (split reduction)
};

struct TileJob {
    int ci, cj;           // C tile (row, col) in tiles
    int a_row0, a_col0;   // global origin of op(A)
    int b_row0, b_col0;   // global origin of op(B)
    int klen;             // length of the reduction
    bool a_trans, b_trans, a_lower, b_lower;
    bool a_sym;           // op(A) is the symmetric matrix A + A^T of a lower tile
    float alpha, beta;
};

// (i, j) of the t-th entry of a row-major enumeration of a lower triangle.
__device__ __forceinline__ void lower_index(int t, int& i, int& j) {
    int r = (int)((sqrt(8.0 * t + 1.0) - 1.0) * 0.5);
    while ((r + 1) * (r + 2) / 2 <= t) ++r;
    while (r * (r + 1) / 2 > t) --r;
    i = r;
    j = t - r * (r + 1) / 2;
}

template <typename T, int MODE>
__device__ __forceinline__ TileJob make_job(const GemmArgs<T>& g, int tile_id) {
    TileJob job{};
    const int Tt = g.tile;
    const int s = g.step;
    if (MODE == GEMM_FWD_TRAIL) {
        int i, j;
        lower_index(tile_id, i, j);
        i += s + 1;
        j += s + 1;
        job.ci = i; job.cj = j;
        job.a_row0 = i * Tt; job.a_col0 = s * Tt; job.a_trans = false;
        job.b_row0 = j * Tt; job.b_col0 = s * Tt; job.b_trans = true;
        job.klen = min(Tt, g.n - s * Tt);
        job.alpha = -1.f; job.beta = 1.f;
    } else if (MODE == GEMM_REV_ROW) {
        const int K = tile_id;  // K <= J = s
        const int r0 = s * Tt + min(Tt, g.n - s * Tt);
        job.ci = s; job.cj = K;
        job.a_row0 = r0; job.a_col0 = s * Tt; job.a_trans = true;
        job.b_row0 = r0; job.b_col0 = K * Tt; job.b_trans = false;
        job.klen = g.n - r0;
        job.alpha = -1.f; job.beta = 1.f;
    } else if (MODE == GEMM_REV_UPD) {
        const int I = s + 1 + tile_id / s, K = tile_id % s;
        job.ci = I; job.cj = K;
        job.a_row0 = I * Tt; job.a_col0 = s * Tt; job.a_trans = false;
        job.b_row0 = s * Tt; job.b_col0 = K * Tt; job.b_trans = false;
        job.klen = min(Tt, g.n - s * Tt);
        job.alpha = -1.f; job.beta = 1.f;
    } else {  // GEMM_REV_SYM
        const int K = tile_id;  // K < J = s
        job.ci = s; job.cj = K;
        job.a_row0 = s * Tt; job.a_col0 = s * Tt; job.a_trans = false; job.a_sym = true;
        job.b_row0 = s * Tt; job.b_col0 = K * Tt; job.b_trans = false;
        job.klen = min(Tt, g.n - s * Tt);
        job.alpha = -1.f; job.beta = 1.f;
    }
    return job;
}

template <typename T, int BM, int MODE>
__global__ void __launch_bounds__(kThreads)
gemm_kernel(GemmArgs<T> g) {
    using R = real_t<T>;
    constexpr int BK = 16;
    constexpr int MT = BM / 16;  // micro-tile per thread (MT x MT)
    constexpr int PAD = sizeof(T) >= 16 ? 1 : 16 / sizeof(T);
    __shared__ __align__(16) T As[BK][BM + PAD];
    __shared__ __align__(16) T Bs[BK][BM + PAD];
    const int subs_per_side = g.tile / BM;
    const int sub = blockIdx.x % (subs_per_side * subs_per_side);
    const int tile_id = blockIdx.x / (subs_per_side * subs_per_side);
    const TileJob job = make_job<T, MODE>(g, tile_id);
    const int r_off = (sub / subs_per_side) * BM;  // sub-block origin inside the tile
    const int c_off = (sub % subs_per_side) * BM;
    const int crow0 = job.ci * g.tile + r_off;
    const int ccol0 = job.cj * g.tile + c_off;
    if (crow0 >= g.n || ccol0 >= g.n) return;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int64_t nn = (int64_t)g.n * g.n;

    for (int64_t b = blockIdx.y; b < g.batch; b += gridDim.y) {
        if (skip_matrix(g.status, b)) continue;
        T* Cb = g.C + b * nn;
        const T* Ab = g.A + b * nn;
        const T* Bb = g.B + b * nn;
        T acc[MT][MT];
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int j = 0; j < MT; ++j) acc[i][j] = T{};

        const int kbeg = blockIdx.z * g.kchunk;
        const int kend = min(job.klen, kbeg + g.kchunk);
        for (int k0 = kbeg; k0 < kend; k0 += BK) {
            __syncthreads();
            // op(A)(r, kk) for r in the sub-block rows, kk in [k0, k0 + BK)
            for (int e = threadIdx.x; e < BK * BM; e += blockDim.x) {
                int r, kk;
                if (job.a_trans) { kk = e / BM; r = e % BM; }   // contiguous over r
                else             { r = e / BK;  kk = e % BK; }  // contiguous over kk
                int gr = job.a_trans ? job.a_row0 + k0 + kk : job.a_row0 + r_off + r;
                int gc = job.a_trans ? job.a_col0 + r_off + r : job.a_col0 + k0 + kk;
                T x = T{};
                if (k0 + kk < kend && gr < g.n && gc < g.n) {
                    if (job.a_sym) {
                        // (A + A^H) of a lower tile: the upper half mirrors the lower
                        // one (conjugated) and the diagonal is doubled
                        const bool diag = gc == gr, upper = gc > gr;
                        if (upper) { const int t = gr; gr = gc; gc = t; }
                        x = Ab[(int64_t)gr * g.n + gc];
                        if (upper) x = conj(x);
                        if (diag) x = add(x, x);
                    } else if (!job.a_lower || gc <= gr) {
                        x = Ab[(int64_t)gr * g.n + gc];
                        if (job.a_trans) x = conj(x);  // a transpose is a conjugate transpose
                    }
                }
                As[kk][r] = x;
            }
            // op(B)(kk, c)
            for (int e = threadIdx.x; e < BK * BM; e += blockDim.x) {
                int c, kk;
                if (job.b_trans) { c = e / BK;  kk = e % BK; }  // contiguous over kk
                else             { kk = e / BM; c = e % BM; }   // contiguous over c
                const int gr = job.b_trans ? job.b_row0 + c_off + c : job.b_row0 + k0 + kk;
                const int gc = job.b_trans ? job.b_col0 + k0 + kk : job.b_col0 + c_off + c;
                T x = T{};
                if (k0 + kk < kend && gr < g.n && gc < g.n && (!job.b_lower || gc <= gr)) {
                    x = Bb[(int64_t)gr * g.n + gc];
                    if (job.b_trans) x = conj(x);
                }
                Bs[kk][c] = x;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                T a[MT], bv[MT];
#pragma unroll
                for (int i = 0; i < MT; ++i) a[i] = As[kk][ty * MT + i];
#pragma unroll
                for (int j = 0; j < MT; ++j) bv[j] = Bs[kk][tx * MT + j];
#pragma unroll
                for (int i = 0; i < MT; ++i)
#pragma unroll
                    for (int j = 0; j < MT; ++j) acc[i][j] = madd(a[i], bv[j], acc[i][j]);
            }
        }
        // epilogue
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int r = crow0 + ty * MT + i;
            if (r >= g.n) continue;
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                const int c = ccol0 + tx * MT + j;
                if (c >= g.n) continue;
                // nothing above the diagonal is written: L stays zero there, and the
                // reverse sweep (which may run on the caller's own buffer) never
                // touches W's upper triangle
                if ((MODE == GEMM_FWD_TRAIL || (MODE == GEMM_REV_ROW && job.ci == job.cj)) && c > r)
                    continue;
                T* cp = Cb + (int64_t)r * g.n + c;
                T v = scale(acc[i][j], R(job.alpha));
                if (g.atomic) {
                    atomic_add(cp, v);
                    continue;
                }
                if (job.beta != 0.f) v = add(v, *cp);
                *cp = v;
            }
        }
    }
}

// Largest tile whose diagonal-tile kernels fit in shared memory: 128 for
// elements of up to 8 bytes, 64 for complex double.
template <typename T> constexpr int max_tile() { return sizeof(T) > 8 ? 64 : 128; }

size_t trsm_smem(int kb, int esize) {
    return ((size_t)(kb + kVecPerBlock) * (kb + 1) + kb) * esize;
}

template <typename T, int MODE>
cudaError_t launch_trsm(const T* L, T* W, const int32_t* status, int64_t batch, int n, int t0,
                        int kb, int v_begin, int v_count, cudaStream_t stream) {
    if (v_count <= 0) return cudaSuccess;
    const size_t smem = trsm_smem(kb, sizeof(T));
    auto kern = trsm_kernel<T, MODE>;
    // raised once per device to the largest size any tile needs
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = allow_smem_once(kern, trsm_smem(max_tile<T>(), sizeof(T)), smem_set);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((v_count + kVecPerBlock - 1) / kVecPerBlock), grid_y(batch));
    kern<<<grid, kThreads, smem, stream>>>(L, W, status, batch, n, t0, kb, v_begin, v_count);
    return cudaGetLastError();
}

template <typename T, int MODE>
cudaError_t launch_gemm(GemmArgs<T> g, int tiles, cudaStream_t stream, int ksplits = 1,
                        int klen = 0) {
    if (tiles <= 0) return cudaSuccess;
    const int bm = g.tile >= 64 ? 64 : 32;
    const int subs = (g.tile / bm) * (g.tile / bm);
    unsigned zdim = 1;
    if (ksplits > 1 && klen > 0) {
        // split the reduction over blockIdx.z; partial sums meet by atomics
        const int per = (klen + ksplits - 1) / ksplits;
        g.kchunk = (per + 15) / 16 * 16;
        zdim = (unsigned)((klen + g.kchunk - 1) / g.kchunk);
        g.atomic = zdim > 1;
    } else {
        g.kchunk = 1 << 30;
        g.atomic = 0;
    }
    dim3 grid((unsigned)(tiles * subs), grid_y(g.batch), zdim);
    if (bm == 64) gemm_kernel<T, 64, MODE><<<grid, kThreads, 0, stream>>>(g);
    else gemm_kernel<T, 32, MODE><<<grid, kThreads, 0, stream>>>(g);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Reverse sweep over one diagonal tile (Murray 2016, unblocked form): on entry
// W_JJ holds the gradient w.r.t. the tile's factor L_JJ (lower), on exit the
// gradient w.r.t. the lower entries of the tile D = A_JJ - R R^T it factored.
// Columns j = kb-1 .. 0 in shared memory, one block per matrix.
// ---------------------------------------------------------------------------
// Packed lower-triangle index (i >= j).
__device__ __forceinline__ int tri(int i, int j) { return i * (i + 1) / 2 + j; }

template <typename T, int THREADS>
__global__ void __launch_bounds__(THREADS)
diag_rev_kernel(const T* __restrict__ L, T* __restrict__ W, const int32_t* __restrict__ status,
                int64_t batch, int n, int j0, int kb) {
    // both tiles packed as lower triangles: kb (kb + 1) elements in all
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* Ls = reinterpret_cast<T*>(smem_raw);
    T* Ws = Ls + (size_t)kb * (kb + 1) / 2;
    const int tid = threadIdx.x;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (skip_matrix(status, b)) continue;
        const T* Lb = L + b * (int64_t)n * n;
        T* Wb = W + b * (int64_t)n * n;
        __syncthreads();
        for (int e = tid; e < kb * kb; e += blockDim.x) {
            const int r = e / kb, c = e % kb;
            if (c > r) continue;
            const int64_t o = (int64_t)(j0 + r) * n + j0 + c;
            Ls[tri(r, c)] = Lb[o];
            Ws[tri(r, c)] = Wb[o];
        }
        __syncthreads();
        chol_tile::potrf_adj<THREADS>(Ls, Ws, kb, chol_tile::PackedLower{});
        for (int e = tid; e < kb * kb; e += blockDim.x) {
            const int r = e / kb, c = e % kb;
            if (c <= r) Wb[(int64_t)(j0 + r) * n + j0 + c] = Ws[tri(r, c)];
        }
    }
}

// dst = tril(src) (zeros above the diagonal), matrices with status != 0 skipped.
template <typename T>
__global__ void __launch_bounds__(kThreads)
lower_copy_kernel(const T* __restrict__ src, T* __restrict__ dst,
                  const int32_t* __restrict__ status, int64_t batch, int n) {
    const int64_t nn = (int64_t)n * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * nn;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = e / nn, w = e % nn;
        if (skip_matrix(status, b)) continue;
        const int i = (int)(w / n), j = (int)(w % n);
        dst[e] = (j <= i) ? src[e] : T{};
    }
}

// On the lower triangle (j <= i): dst_ij += src_ij (accumulate; matrices with
// status != 0 skipped), or dst_ij = src_ij (matrices with status != 0 get 0).
template <typename T>
__global__ void __launch_bounds__(kThreads)
lower_add_kernel(const T* __restrict__ src, T* __restrict__ dst,
                 const int32_t* __restrict__ status, int64_t batch, int n, bool accumulate) {
    const int64_t nn = (int64_t)n * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * nn;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = e / nn, w = e % nn;
        const int i = (int)(w / n), j = (int)(w % n);
        if (j > i) continue;
        const bool skip = skip_matrix(status, b);
        if (accumulate) {
            if (!skip) dst[e] = add(dst[e], src[e]);
        } else {
            dst[e] = skip ? T{} : src[e];
        }
    }
}

// Lower triangle of every matrix with status != 0 set to zero (the in-place
// adjoint's rule for skipped matrices); nothing else is touched.
template <typename T>
__global__ void __launch_bounds__(kThreads)
zero_lower_skipped_kernel(T* __restrict__ dst, const int32_t* __restrict__ status, int64_t batch,
                          int n) {
    const int64_t nn = (int64_t)n * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * nn;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = e / nn, w = e % nn;
        const int i = (int)(w / n), j = (int)(w % n);
        if (j <= i && skip_matrix(status, b)) dst[e] = T{};
    }
}

inline unsigned elementwise_blocks(int64_t total) {
    return (unsigned)std::max<int64_t>(
        1, std::min<int64_t>((total + kThreads - 1) / kThreads, (int64_t)device_sm_count() * 16));
}

}  // namespace

// Large matrices take 128-wide tiles (fewer, longer GEMMs); below that, 64
// when the batch alone gives every SM several 64-wide tiles to work on, else
// 32 so that a few matrices still spread over the GPU.
int blocked_default_tile(int n, int64_t batch) {
    if (n >= 2048) return 128;
    const int64_t per_side = (n + 63) / 64;
    return batch * per_side * per_side >= 4 * (int64_t)device_sm_count() ? 64 : 32;
}

#define CHOL_TRY(x)                              \
    do {                                         \
        cudaError_t e_ = (x);                    \
        if (e_ != cudaSuccess) return e_;        \
    } while (0)

size_t blocked_fwd_workspace_bytes(bool real_double, int64_t batch, int n, int tile) {
    if (!real_double || tile != 128 || n <= 128) return 0;
    return ozaki_workspace_bytes(batch, n);
}

template <typename T>
cudaError_t blocked_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n, int tile,
                        void* work, cudaStream_t stream) {
    const int nt = (n + tile - 1) / tile;
    {
        const int64_t total = batch * (int64_t)n * n;
        const int64_t blocks =
            std::min<int64_t>((total + kThreads - 1) / kThreads, (int64_t)device_sm_count() * 32);
        tril_copy_kernel<T><<<(unsigned)std::max<int64_t>(blocks, 1), kThreads, 0, stream>>>(
            A, L, status, batch, n);
        CHOL_TRY(cudaGetLastError());
    }
    static std::atomic<uint64_t> diag_smem_set{0};
    CHOL_TRY(allow_smem_once(potrf_diag_kernel<T, kThreads>,
                             (size_t)max_tile<T>() * (max_tile<T>() + 1) * sizeof(T),
                             diag_smem_set));
    // float64, 128-wide tiles, workspace: the tensor-core path, with lookahead
    // on a side stream when there are at least three tile columns and the
    // caller's stream is not being captured into a graph
    const bool oz = std::is_same<T, double>::value && work != nullptr && tile == 128;
    SideStream sd;
    int dev = 0;
    bool look = false;
    if (oz && nt >= 3) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        const bool idle = cudaStreamIsCapturing(stream, &cap) == cudaSuccess &&
                          cap == cudaStreamCaptureStatusNone;
        cudaGetLastError();
        look = idle && side_stream(dev, sd);
    }
    std::unique_lock<std::mutex> side_lock;
    if (look) side_lock = std::unique_lock<std::mutex>(g_side_lock[dev]);
    JoinSide join{stream, stream, &sd};
    CHOL_TRY(join.start(look));
    const cudaStream_t cs = join.chain;  // the chain's stream
    for (int k = 0; k < nt; ++k) {
        const int k0 = k * tile;
        const int kb = std::min(tile, n - k0);
        // small tiles: two warps, so the per-column barriers stay cheap
        const size_t dsm = (size_t)kb * (kb + 1) * sizeof(T);
        bool on_cluster = false;
        if constexpr (std::is_same<T, double>::value || std::is_same<T, float>::value) {
            if (cluster_diag_pays(batch, kb)) {
                // few matrices: the tile on a cluster of SMs, which for the
                // tensor-core panel solve also inverts it
                T* inv = nullptr;
                int32_t* bal = nullptr;
                if constexpr (std::is_same<T, double>::value) {
                    if (oz && k < nt - 1) {
                        double* id = nullptr;
                        ozaki_fwd_inverse(work, batch, n, &id, &bal);
                        inv = id;
                    }
                }
                CHOL_TRY(cluster_potrf_diag(L, status, batch, n, k0, kb, inv, bal, cs));
                on_cluster = true;
            }
        }
        if (on_cluster) {
        } else if (kb <= 32)
            potrf_diag_kernel<T, 64><<<dim3(1, grid_y(batch)), 64, dsm, cs>>>(L, status, batch,
                                                                                 n, k0, kb);
        else
            potrf_diag_kernel<T, kThreads><<<dim3(1, grid_y(batch)), kThreads, dsm, cs>>>(
                L, status, batch, n, k0, kb);
        CHOL_TRY(cudaGetLastError());
        if (k == nt - 1) break;
        if constexpr (std::is_same<T, double>::value) {
            if (oz) {
                // panel solve and trailing update on the tensor cores
                double* Ld = reinterpret_cast<double*>(L);
                CHOL_TRY(ozaki_panel_solve(Ld, work, status, batch, n, k, on_cluster, cs));
                CHOL_TRY(ozaki_trailing_slice(Ld, work, status, batch, n, k, cs));
                if (!look) {
                    CHOL_TRY(ozaki_trailing_gemm(Ld, work, status, batch, n, k, 0, cs));
                    continue;
                }
                // block column k + 1 here (the last step's remaining columns,
                // which include it, first); the columns right of it on the
                // side stream, beside the next step's factor and panel solve
                if (join.pending) {
                    CHOL_TRY(cudaStreamWaitEvent(cs, sd.rest, 0));
                    join.pending = false;
                }
                CHOL_TRY(ozaki_trailing_gemm(Ld, work, status, batch, n, k, 1, cs));
                if (nt - k - 1 >= 2) {
                    CHOL_TRY(cudaEventRecord(sd.look, cs));
                    CHOL_TRY(cudaStreamWaitEvent(sd.s, sd.look, 0));
                    CHOL_TRY(ozaki_trailing_gemm(Ld, work, status, batch, n, k, 2, sd.s));
                    CHOL_TRY(cudaEventRecord(sd.rest, sd.s));
                    join.pending = true;
                }
                continue;
            }
        }
        CHOL_TRY((launch_trsm<T, TRSM_FWD_PANEL>(L, L, status, batch, n, k0, kb, k0 + kb,
                                                 n - k0 - kb, cs)));
        const int m = nt - k - 1;
        GemmArgs<T> g{L, L, L, status, batch, n, tile, nt, k, 0, 0};
        CHOL_TRY((launch_gemm<T, GEMM_FWD_TRAIL>(g, m * (m + 1) / 2, cs)));
    }
    return join.finish();
}

// Adjoint by the blocked reverse sweep of Murray (2016) over a left-looking
// blocked factorisation, in place on W (= tril(adj_L) on entry):
// for tile columns J = nt-1 .. 0, with C = W's panel below the diagonal tile,
//   C      <- C L_JJ^-1                 (triangular solve, rows of the panel)
//   W_JK   -= C^T L_panel,K   (K <= J)  (reduction over the rows below J)
//   W_IK   -= C L_JK          (I > J, K < J)
//   W_JJ   <- reverse sweep of the tile's own factorisation
//   W_JK   -= (W_JJ + W_JJ^T) L_JK      (K < J)
// and finally adj_A += tril(W).  This is the same lower-triangle gradient as
// Phi(M + M^T), M = L^-T Phi(L^T adj_L) L^-1, in 2 n^3 / 3 flops instead of
// the 7 n^3 / 3 of forming P and solving twice.
template <typename T>
cudaError_t blocked_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status,
                        int64_t batch, int n, int tile, T* W, bool accumulate, void* oz_work,
                        cudaStream_t stream) {
    const int nt = (n + tile - 1) / tile;
    const int64_t total = batch * (int64_t)n * n;
    // In place (the gradient written over its seed): the sweep runs on the
    // caller's buffer itself, whose lower triangle already holds adj_L; no
    // stage reads or writes its upper triangle, so no workspace is needed.
    const bool in_place = !accumulate && Lbar == Abar;
    if (in_place) {
        W = Abar;
    } else {
        lower_copy_kernel<T><<<elementwise_blocks(total), kThreads, 0, stream>>>(Lbar, W, status,
                                                                                batch, n);
        CHOL_TRY(cudaGetLastError());
    }
    static std::atomic<uint64_t> diag_smem_set{0};
    CHOL_TRY(allow_smem_once(diag_rev_kernel<T, kThreads>,
                             (size_t)max_tile<T>() * (max_tile<T>() + 1) * sizeof(T),
                             diag_smem_set));
    const int sms = device_sm_count();
    const int bm = tile >= 64 ? 64 : 32;
    const int subs = (tile / bm) * (tile / bm);
    const int64_t bmat = std::min<int64_t>(batch, 65535);
    // float64 with 128-wide tiles: the two large updates on the tensor cores
    bool oz = false;
    if constexpr (std::is_same<T, double>::value) {
        oz = oz_work != nullptr && tile == 128;
        if (oz) CHOL_TRY(ozaki_adj_prepare(L, oz_work, status, batch, n, stream));
    }
    // lookahead (as in the forward): tile column J's row update and update of
    // block columns J - 1 .. J here, of the columns left of those on the side
    // stream, beside tile column J - 1's solve, row update and diagonal tile
    SideStream sd;
    int dev = 0;
    bool look = false;
    if (oz && nt >= 3) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        const bool idle = cudaStreamIsCapturing(stream, &cap) == cudaSuccess &&
                          cap == cudaStreamCaptureStatusNone;
        cudaGetLastError();
        look = idle && side_stream(dev, sd);
    }
    std::unique_lock<std::mutex> side_lock;
    if (look) side_lock = std::unique_lock<std::mutex>(g_side_lock[dev]);
    JoinSide join{stream, stream, &sd};
    CHOL_TRY(join.start(look));
    const cudaStream_t cs = join.chain;  // the chain's stream
    for (int J = nt - 1; J >= 0; --J) {
        const int j0 = J * tile, kb = std::min(tile, n - j0), r0 = j0 + kb, nb = n - r0;
        if constexpr (std::is_same<T, double>::value) {
            if (oz) {
                // with lookahead the row update's block columns K < J - 1 go to
                // the side stream (below), after the update of column J - 1
                const bool split_row = look && J >= 2;
                if (nb > 0) {
                    CHOL_TRY(ozaki_adj_solve(L, W, oz_work, status, batch, n, J, cs));
                    CHOL_TRY(ozaki_adj_row(L, W, oz_work, status, batch, n, J, split_row ? 1 : 0,
                                           cs));
                }
                if (ozaki_adj_lit_pays(batch)) {
                    // few matrices: the tile's adjoint as three parallel products
                    CHOL_TRY(ozaki_adj_diag(L, W, oz_work, status, batch, n, J, cs));
                } else {
                    const size_t dsm = (size_t)kb * (kb + 1) * sizeof(T);
                    diag_rev_kernel<T, kThreads><<<dim3(1, grid_y(batch)), kThreads, dsm,
                                                   cs>>>(L, W, status, batch, n, j0, kb);
                    CHOL_TRY(cudaGetLastError());
                }
                // W_IK -= C_I L_JK (I > J) and W_JK -= (W_JJ + W_JJ^T) L_JK, K < J
                if (J == 0) continue;
                double* Wd = reinterpret_cast<double*>(W);
                CHOL_TRY(ozaki_adj_upd_slice(Wd, oz_work, status, batch, n, J, cs));
                if (!look) {
                    CHOL_TRY(ozaki_adj_upd_gemm(Wd, oz_work, status, batch, n, J, 0, cs));
                    continue;
                }
                if (join.pending) {
                    CHOL_TRY(cudaStreamWaitEvent(cs, sd.rest, 0));
                    join.pending = false;
                }
                CHOL_TRY(ozaki_adj_upd_gemm(Wd, oz_work, status, batch, n, J, 1, cs));
                if (J >= 2) {
                    CHOL_TRY(cudaEventRecord(sd.look, cs));
                    CHOL_TRY(cudaStreamWaitEvent(sd.s, sd.look, 0));
                    if (split_row && nb > 0)
                        CHOL_TRY(ozaki_adj_row(L, W, oz_work, status, batch, n, J, 2, sd.s));
                    CHOL_TRY(ozaki_adj_upd_gemm(Wd, oz_work, status, batch, n, J, 2, sd.s));
                    CHOL_TRY(cudaEventRecord(sd.rest, sd.s));
                    join.pending = true;
                }
                continue;
            }
        }
        if (nb > 0) {
            CHOL_TRY((launch_trsm<T, TRSM_ADJ_M>(L, W, status, batch, n, j0, kb, r0, nb, cs)));
            GemmArgs<T> g{W, L, W, status, batch, n, tile, nt, J, 0, 0};
            // enough blocks to fill the GPU twice over, splitting the long reduction
            const int64_t blocks = (int64_t)(J + 1) * subs * bmat;
            const int ks = (int)std::max<int64_t>(
                1, std::min<int64_t>((2 * sms + blocks - 1) / blocks, (nb + 127) / 128));
            CHOL_TRY((launch_gemm<T, GEMM_REV_ROW>(g, J + 1, cs, ks, nb)));
            if (J > 0) CHOL_TRY((launch_gemm<T, GEMM_REV_UPD>(g, (nt - J - 1) * J, cs)));
        }
        const size_t dsm = (size_t)kb * (kb + 1) * sizeof(T);
        if (kb <= 32)
            diag_rev_kernel<T, 64><<<dim3(1, grid_y(batch)), 64, dsm, cs>>>(L, W, status, batch,
                                                                              n, j0, kb);
        else
            diag_rev_kernel<T, kThreads><<<dim3(1, grid_y(batch)), kThreads, dsm, cs>>>(
                L, W, status, batch, n, j0, kb);
        CHOL_TRY(cudaGetLastError());
        if (J > 0) {
            GemmArgs<T> g{W, L, W, status, batch, n, tile, nt, J, 0, 0};
            CHOL_TRY((launch_gemm<T, GEMM_REV_SYM>(g, J, cs)));
        }
    }
    // the chain and the side stream's last update land before W is read below
    CHOL_TRY(join.finish());
    if (in_place) {
        if (status != nullptr)
            zero_lower_skipped_kernel<T><<<elementwise_blocks(total), kThreads, 0, stream>>>(
                Abar, status, batch, n);
    } else {
        lower_add_kernel<T><<<elementwise_blocks(total), kThreads, 0, stream>>>(W, Abar, status,
                                                                               batch, n, accumulate);
    }
    return cudaGetLastError();
}

template cudaError_t blocked_fwd<float>(const float*, float*, int32_t*, int64_t, int, int, void*,
                                        cudaStream_t);
template cudaError_t blocked_fwd<double>(const double*, double*, int32_t*, int64_t, int, int,
                                         void*, cudaStream_t);
template cudaError_t blocked_adj<float>(const float*, const float*, float*, const int32_t*,
                                        int64_t, int, int, float*, bool, void*, cudaStream_t);
template cudaError_t blocked_adj<double>(const double*, const double*, double*, const int32_t*,
                                         int64_t, int, int, double*, bool, void*, cudaStream_t);
template cudaError_t blocked_fwd<cplx<float>>(const cplx<float>*, cplx<float>*, int32_t*, int64_t,
                                              int, int, void*, cudaStream_t);
template cudaError_t blocked_fwd<cplx<double>>(const cplx<double>*, cplx<double>*, int32_t*,
                                               int64_t, int, int, void*, cudaStream_t);
template cudaError_t blocked_adj<cplx<float>>(const cplx<float>*, const cplx<float>*, cplx<float>*,
                                              const int32_t*, int64_t, int, int, cplx<float>*, bool,
                                              void*, cudaStream_t);
template cudaError_t blocked_adj<cplx<double>>(const cplx<double>*, const cplx<double>*,
                                               cplx<double>*, const int32_t*, int64_t, int, int,
                                               cplx<double>*, bool, void*, cudaStream_t);

}  // namespace chol
