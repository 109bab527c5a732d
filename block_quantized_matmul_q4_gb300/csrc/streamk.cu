// streamk.cu -- grid size, partial area and fixup of the stream-K GEMMs
// (gemm_f16.cu). With more tiles than SMs, a persistent grid of
// one CTA per SM takes the units u = tile * nsb + k-round in equal
// contiguous ranges (CTA c: [c U / G, (c+1) U / G)); a CTA that holds all of
// a tile's units writes it, otherwise its piece went to its partial slot
// (slot 0 when the tile is the CTA's first, 1 when its last), fp32
// [G][2][TN cols][128 rows]. Here every split tile gets the sum of its
// pieces, added in CTA order (the same order every run), written to C.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kTM = kSkTile;  // tile rows (weights); TN, the columns (tokens), is a template parameter
constexpr int64_t kMaxGrid = 1024;           // CTAs of a persistent grid at most
constexpr int kFixupThreads = 512;

int64_t max_grid() {
    const int64_t n = sm_count();
    return n < kMaxGrid ? n : kMaxGrid;
}

template <class T>
__device__ __forceinline__ T out_cast(float v);
template <>
__device__ __forceinline__ float out_cast<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half out_cast<__half>(float v) { return __float2half_rn(v); }

// Rows n .. n+3 of one column of C in a single store (C's rows 16-byte
// aligned for fp32, 8-byte for fp16, n a multiple of 4).
__device__ __forceinline__ void store4(float *y, float4 v) { *reinterpret_cast<float4 *>(y) = v; }
__device__ __forceinline__ void store4(__half *y, float4 v) {
    const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(y) = make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                                               *reinterpret_cast<const uint32_t *>(&hi));
}

// The pieces of one split tile added in CTA order and stored, by `splits`
// CTAs per tile, each over TN / splits of its columns: for split-K grids
// (fewer tiles than half the SMs, each tile in many pieces) enough CTAs for
// about two per SM, so that the few tiles still spread over all the SMs; for
// stream-K grids (a tile in two or three pieces) one CTA per tile. Each thread takes 4
// consecutive rows of a column (a 16-byte load per piece), kQ of them, and
// issues the loads of up to kBatch pieces before adding them, in CTA order
// (the same order every run). A warp covers 128 rows of one column = 512
// contiguous bytes of every slot. Columns past the last token (rounded up to
// 16, the columns the GEMM epilogue wrote) are skipped. vec: C's rows are
// aligned for one 4-row store (N a multiple of 4, C aligned).
// kFixupQ quads per thread, kFixupBatch pieces loaded at once: 2 x 4 for
// split-K (many pieces, two CTAs per SM), 4 x 2 for stream-K (two or three
// pieces, one CTA per tile: eight loads in flight per thread).
template <int TN, class T, int kFixupQ, int kFixupBatch>
__global__ void __launch_bounds__(kFixupThreads, kFixupQ == 2 ? 2 : 1) fixup_kernel(const float *__restrict__ part,
                                                                       T *__restrict__ C, int64_t N,
                                                                       int64_t M, int64_t mblocks,
                                                                       int64_t nsb, int64_t units,
                                                                       int64_t G, int splits, bool vec) {
    pdl_wait();  // the GEMM's pieces
    const int64_t tile = blockIdx.x / splits;
    const int split = (int)(blockIdx.x % splits);
    const int64_t ca = sk_cta_of(tile * nsb, units, G), cb = sk_cta_of(tile * nsb + nsb - 1, units, G);
    if (ca == cb) return;  // written whole by its CTA
    // Slots of the pieces, without a division per piece: every CTA after ca
    // starts inside the tile (its first tile: slot 0); ca's piece is in slot 0
    // only when ca's range starts at the tile, else in slot 1 (its last tile).
    const int64_t sbytes = (int64_t)kTM * TN;
    const int64_t slot_ca = (ca * 2 + (ca * units / G < tile * nsb ? 1 : 0)) * sbytes;
    const int64_t n0 = (tile / mblocks) * kTM, m0 = (tile % mblocks) * TN;
    const int64_t mv = M - m0 < TN ? M - m0 : TN;  // columns holding tokens
    const int cols = TN / splits, c0 = split * cols;
    const int cend = (int)((mv + 15) / 16 * 16) < c0 + cols ? (int)((mv + 15) / 16 * 16) : c0 + cols;
    const int nquads = (cend - c0) * (kTM / 4);
    for (int e0 = threadIdx.x; e0 < nquads; e0 += kFixupQ * kFixupThreads) {
        float4 v[kFixupQ];
        int rr[kFixupQ], cc[kFixupQ];
        bool live[kFixupQ];
#pragma unroll
        for (int h = 0; h < kFixupQ; ++h) {
            const int e = e0 + h * kFixupThreads;
            live[h] = e < nquads;
            rr[h] = (e % (kTM / 4)) * 4;
            cc[h] = c0 + e / (kTM / 4);
            v[h] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        for (int64_t k0 = ca; k0 <= cb; k0 += kFixupBatch) {
            float4 p[kFixupBatch][kFixupQ];
#pragma unroll
            for (int b = 0; b < kFixupBatch; ++b) {
                if (k0 + b > cb) break;
                const float *slot = part + (k0 + b == ca ? slot_ca : (k0 + b) * 2 * sbytes);
#pragma unroll
                for (int h = 0; h < kFixupQ; ++h)
                    if (live[h]) p[b][h] = __ldcg(reinterpret_cast<const float4 *>(slot + cc[h] * kTM + rr[h]));
            }
#pragma unroll
            for (int b = 0; b < kFixupBatch; ++b) {
                if (k0 + b > cb) break;
#pragma unroll
                for (int h = 0; h < kFixupQ; ++h) {
                    if (!live[h]) continue;
                    if (k0 + b == ca) {
                        v[h] = p[b][h];
                    } else {
                        v[h].x += p[b][h].x;
                        v[h].y += p[b][h].y;
                        v[h].z += p[b][h].z;
                        v[h].w += p[b][h].w;
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < kFixupQ; ++h) {
            const int64_t m = m0 + cc[h], n = n0 + rr[h];
            if (live[h] && m < M) {
                T *y = C + m * N + n;
                if (vec && n + 3 < N) {
                    store4(y, v[h]);
                    continue;
                }
                if (n < N) y[0] = out_cast<T>(v[h].x);
                if (n + 1 < N) y[1] = out_cast<T>(v[h].y);
                if (n + 2 < N) y[2] = out_cast<T>(v[h].z);
                if (n + 3 < N) y[3] = out_cast<T>(v[h].w);
            }
        }
    }
}

}  // namespace

// Grid of the stream-K GEMMs for `tiles` output tiles of `units` (tile,
// round) units: one CTA per SM when tiles outnumber SMs; one CTA per tile
// from half the SM count up (no split: measured no faster split than whole
// at 128 tiles); below that the units of the few tiles spread over the SMs
// (split K), which the same piece/fixup machinery sums.
int64_t stream_k_grid(int64_t tiles, int64_t units) {
    const int64_t g = max_grid();
    if (tiles > g) return g;
    if (2 * tiles >= g) return tiles < 1 ? 1 : tiles;
    return units < g ? (units < 1 ? 1 : units) : g;
}

bool stream_k_splits(int wt, int64_t N, int64_t M, int64_t K) {
    const int64_t tn = gemm_tile_cols(wt, M);
    const int64_t tiles = ((N + kTM - 1) / kTM) * ((M + tn - 1) / tn);
    const int64_t units = tiles * ((K + kSkRound - 1) / kSkRound);
    return stream_k_grid(tiles, units) != tiles;
}

// Two fp32 slots of the widest tile per CTA of the largest grid.
size_t stream_k_part_bytes() { return align_up((size_t)2 * max_grid() * kTM * kSkColsMax * 4, 256); }

template <int TN>
cudaError_t launch_fixup_tn(const float *part, void *C, bool half_out, int64_t N, int64_t M, int64_t mblocks,
                            int64_t nsb, int64_t units, int64_t G, cudaStream_t s) {
    const int64_t nblocks = (N + kTM - 1) / kTM, tiles = nblocks * mblocks;
    // CTAs per tile: enough for about two per SM over all tiles, a power of
    // two up to one per 32 columns
    const bool split_k = tiles < G;  // else stream-K: one CTA per tile, four quads per thread
    int splits = 1;
    while (split_k && splits < TN / 32 && tiles * splits < 2 * (int64_t)sm_count()) splits *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * splits));
    cfg.blockDim = dim3(kFixupThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool vh = N % 4 == 0 && (uintptr_t)C % 8 == 0, vf = N % 4 == 0 && (uintptr_t)C % 16 == 0;
    if (!split_k)
        return half_out ? cudaLaunchKernelEx(&cfg, fixup_kernel<TN, __half, 4, 2>, part,
                                             static_cast<__half *>(C), N, M, mblocks, nsb, units, G, 1, vh)
                        : cudaLaunchKernelEx(&cfg, fixup_kernel<TN, float, 4, 2>, part,
                                             static_cast<float *>(C), N, M, mblocks, nsb, units, G, 1, vf);
    return half_out ? cudaLaunchKernelEx(&cfg, fixup_kernel<TN, __half, 2, 4>, part, static_cast<__half *>(C),
                                         N, M, mblocks, nsb, units, G, splits, vh)
                    : cudaLaunchKernelEx(&cfg, fixup_kernel<TN, float, 2, 4>, part, static_cast<float *>(C), N,
                                         M, mblocks, nsb, units, G, splits, vf);
}

cudaError_t launch_stream_k_fixup(const float *part, void *C, bool half_out, int cols, int64_t N, int64_t M,
                                  int64_t mblocks, int64_t nsb, int64_t units, int64_t G,
                                  cudaStream_t s) {
    cudaError_t e = cols == 256 ? launch_fixup_tn<256>(part, C, half_out, N, M, mblocks, nsb, units, G, s)
                                : launch_fixup_tn<128>(part, C, half_out, N, M, mblocks, nsb, units, G, s);
    count_launch();
    return e;
}

}  // namespace qmm
