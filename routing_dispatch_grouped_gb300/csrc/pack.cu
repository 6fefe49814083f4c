// One-time repacking of expert weights into the tile-contiguous layout the grouped GEMMs stream
// fastest (a storage layout of this library; the pages' layout stays the input format).
//
// The pages' layout ("Tensor parallelism for inference", "Packed strategies": gate_up_proj
// [E, hidden, 2*expert_dim], gate first; down [E, expert_dim, hidden]) makes every 64-column x
// 64-row weight tile the GEMMs load a set of 64 rows of 128 bytes, one full weight row apart.
// Packed, each such tile is one contiguous 8 KB block, so streaming an expert's weights reads
// memory sequentially:
//   block (e, nb, kb) = rows k in [64 kb, 64 kb + 64) of columns [64 c, 64 c + 64), stored at
//   rows ((e * NB + nb) * Kpad + k) of a [E * NB * Kpad, 64] matrix, Kpad = K rounded up to 64.
//   down:    NB = ceil(N / 64), block nb holds columns [64 nb, 64 nb + 64).
//   gate_up: the gate half and the up half are blocked separately, NBh = ceil(I / 64) blocks
//            each (NB = 2 NBh); block nb < NBh holds gate columns [64 nb, ...), block NBh + j
//            holds up columns [64 j, ...) (column I + 64 j of the pages' layout).
// Padding rows and columns are zero, so the GEMMs' K loop may run over Kpad.
#include "moe_internal.cuh"

namespace rdg {
namespace {

__global__ void __launch_bounds__(256) pack_kernel(const uint4* __restrict__ w,
                                                   uint4* __restrict__ packed, long long n_vec,
                                                   int K, int n_cols, int row_cols, int nb,
                                                   int nbh, int kpad, int halves) {
    griddep_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += stride) {
        const long long r = v >> 3;          // packed row
        const int c8 = (int)(v & 7);         // 8-column group inside the 64-column block
        const int k = (int)(r % kpad);
        const long long eb = r / kpad;
        const int blk = (int)(eb % nb);
        const long long e = eb / nb;
        int half = 0, cb = blk;
        if (halves == 2) {
            half = blk / nbh;
            cb = blk - half * nbh;
        }
        const int col = cb * 64 + c8 * 8;    // column within the half (or the whole matrix)
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (k < K && col < n_cols)
            val = __ldg(w + ((e * K + k) * (long long)row_cols + (long long)half * n_cols + col) / 8);
        packed[v] = val;
    }
}

}  // namespace

PackedGeom packed_geom(int kind, int K, int N) {
    PackedGeom g;
    g.kpad = (K + kTileK - 1) / kTileK * kTileK;
    g.nbh = (N + 63) / 64;
    g.nb = (kind == kGateUp) ? 2 * g.nbh : g.nbh;
    return g;
}

cudaError_t launch_pack_weights(int kind, const void* w, void* packed, int E, int K, int N,
                                cudaStream_t s) {
    const PackedGeom g = packed_geom(kind, K, N);
    const long long rows = (long long)E * g.nb * g.kpad;
    const long long n_vec = rows * 8;  // 16-byte vectors: 8 per 64-column row
    const int row_cols = (kind == kGateUp) ? 2 * N : N;
    long long blocks = (n_vec + 255) / 256;
    const long long cap = (long long)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_kernel(pack_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                         static_cast<const uint4*>(w), static_cast<uint4*>(packed), n_vec, K, N,
                         row_cols, g.nb, g.nbh, g.kpad, kind == kGateUp ? 2 : 1);
}

}  // namespace rdg
