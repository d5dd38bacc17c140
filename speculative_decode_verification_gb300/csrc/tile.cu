// tile.cu - conversion of row-major affine Q4/g64 weights into the library's
// tiled layout (q4_tile in include/verify.h).
//
// The tiled layout stores each (128-row tile, chunk of G 64-column groups) of
// a matrix as one contiguous block, in exactly the order the verify kernels
// keep it in shared memory, so that one bulk copy moves a pipeline stage and
// HBM is read in long contiguous runs:
//
//   block = [scales: 128 rows x G groups bf16][biases: same]     512 G bytes
//           [codes of group 0][codes of group 1] ... (gcount)    4096 each
//
// G = 4 (256-column chunks) for dense products; G = 2 (128-column chunks)
// for the routed and shared experts' gate/up and down matrices.
//
// Codes of one group (64 columns of 128 rows) are ordered for the MMA
// fragments: for 16-row block b (0..7) and lane L = 4g + c (0..31), 16 bytes =
// the words {row 16b+g: W0, row 16b+g+8: W0, row 16b+g: W1, row 16b+g+8: W1},
// where W0 / W1 hold columns 16c .. 16c+7 / 16c+8 .. 16c+15 of the group with
// the nibble at position p taken from column 16c + 8w + sigma(p),
// sigma = (0 4 2 6 1 5 3 7): decoding nibble pair (p, p+4) of such a word
// gives the bf16 pair the m16n8k16 A fragment wants for the activation
// columns in their natural order.
//
// Rows past the matrix are zero (codes, scales and biases).  The last chunk of
// a row holds only the groups that exist (gcount = min(G, K/64 - G kc)); the
// other chunks are 512 G + 4096 G bytes.  A row tile takes 512 G KC + 4096 KG
// bytes (KC = ceil(K/64 / G) chunks).
// With the gate/up pairing, tile t of an expert holds gate rows 64t .. 64t+63
// then up rows I + 64t .. I + 64t + 63 (I = n_out / 2).
#include "common.cuh"
#include "internal.h"

namespace vk {

__device__ __forceinline__ uint32_t sigma_nibbles(uint32_t u) {
  constexpr int sigma[8] = {0, 4, 2, 6, 1, 5, 3, 7};
  uint32_t out = 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) out |= ((u >> (4 * sigma[p])) & 0xFu) << (4 * p);
  return out;
}

// One block per (expert, row tile, chunk), 256 threads; GR groups per chunk.
__global__ void __launch_bounds__(256) tile_kernel(const uint32_t* packed, const uint16_t* scales,
                                                   const uint16_t* biases, uint8_t* dst, int N, int K, int gate_up,
                                                   int GR) {
  const int KG = K / 64, KC = (KG + GR - 1) / GR, KW = K / 8;
  const int RT = gate_up ? N / kBM : (N + kBM - 1) / kBM;
  long long b = blockIdx.x;
  const int kc = (int)(b % KC);
  b /= KC;
  const int rt = (int)(b % RT);
  const long long e = b / RT;
  const long long rt_bytes = tile_row_bytes(K, GR);
  const int sb_bytes = tile_sb_bytes(GR);
  uint8_t* blk = dst + (e * RT + rt) * rt_bytes + (long long)kc * tile_chunk_bytes(GR);
  const int gcount = min(GR, KG - GR * kc);
  const uint32_t* P = packed + e * N * KW;
  const uint16_t* Sc = scales + e * N * KG;
  const uint16_t* Bi = biases + e * N * KG;
  auto mrow = [&](int i) -> int {
    if (gate_up) return i < 64 ? 64 * rt + i : N / 2 + 64 * rt + (i - 64);
    const int r = rt * kBM + i;
    return r < N ? r : -1;
  };
  const int t = threadIdx.x;
  // scales then biases, [row][GR groups] bf16 each (GR = 2 or 4)
  for (int i = t; i < kBM * GR; i += blockDim.x) {
    const int row = i / GR, G = i % GR;
    const int r = mrow(row);
    const bool ok = r >= 0 && G < gcount;
    reinterpret_cast<uint16_t*>(blk)[i] = ok ? Sc[(long long)r * KG + GR * kc + G] : (uint16_t)0;
    reinterpret_cast<uint16_t*>(blk + sb_bytes / 2)[i] = ok ? Bi[(long long)r * KG + GR * kc + G] : (uint16_t)0;
  }
  const int bk = t >> 5, lane = t & 31, g = lane >> 2, c = lane & 3;
  const int r0 = mrow(16 * bk + g), r1 = mrow(16 * bk + g + 8);
  for (int G = 0; G < gcount; ++G) {
    const long long wi = 8LL * (GR * kc + G) + 2 * c;
    const uint32_t u0 = r0 >= 0 ? P[(long long)r0 * KW + wi] : 0u, u1 = r0 >= 0 ? P[(long long)r0 * KW + wi + 1] : 0u;
    const uint32_t u2 = r1 >= 0 ? P[(long long)r1 * KW + wi] : 0u, u3 = r1 >= 0 ? P[(long long)r1 * KW + wi + 1] : 0u;
    *reinterpret_cast<uint4*>(blk + sb_bytes + ((G * 8 + bk) * 32 + lane) * 16) =
        make_uint4(sigma_nibbles(u0), sigma_nibbles(u2), sigma_nibbles(u1), sigma_nibbles(u3));
  }
}

static int kind_groups(int kind) { return kind == 0 ? kGroupsPerUnit : kExpertGroups; }

long long tiled_bytes(int N, int K, int E, int kind) {
  const long long RT = kind == 1 ? N / kBM : (N + kBM - 1) / kBM;
  return (long long)E * RT * tile_row_bytes(K, kind_groups(kind));
}

cudaError_t launch_tile(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases, uint8_t* dst, int N,
                        int K, int E, int kind, cudaStream_t s) {
  const int GR = kind_groups(kind);
  const long long KG = K / 64, KC = (KG + GR - 1) / GR;
  const long long RT = kind == 1 ? N / kBM : (N + kBM - 1) / kBM;
  const long long blocks = (long long)E * RT * KC;
  if (blocks <= 0 || blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  tile_kernel<<<(unsigned)blocks, 256, 0, s>>>(packed, scales, biases, dst, N, K, kind == 1 ? 1 : 0, GR);
  return cudaGetLastError();
}

}  // namespace vk
