// Host-side choice of the pair GEMM's tile shape (the kernels in gemm_pair.cu are built for these shapes),
// kept apart from the kernels so that a change of policy leaves the kernel source untouched.
#include "kernels.h"

namespace lynx {

// Shared-memory traffic per thousand logical MACs of each sparse shape (TMA fill plus tensor-core operand
// reads, the kernel's binding resource): 512 x 224 tiles 21.3 B, 512 x 192 tiles 22.9 B, 256 x 256 tiles
// 23.8 B, 256 x 192 tiles 26.7 B.  The shape with the smallest (tile waves x tile work x traffic) wins: 512 x 224
// for the large DiT QKV and MLP-up shapes, 512 x 192 where 224-wide column tiles would add a wave (N = 3072),
// 256 x 256 when few row tiles would leave pairs idle (e.g. M = 1024, N = 9216), 256 x 192 when narrower tiles
// keep a short problem inside one wave (e.g. M = 1024, N = 3072: 64 tiles for 76 CTA pairs).
// Dense shapes: the 256 x 448 tile does a tile's work in 0.965 of the time of 1.75 256 x 256 tiles (measured at
// M = 4608-16384, K = 3072), so it wins where its waves are about as full as the 256-column tiles' (QKV N = 9216:
// 5 waves instead of 9, 0.95x the time; N = 3072 at M = 16384: 0.87x) and loses where a wave stays partly idle
// (N = 3072 at M = 4608: 2 waves of 126 tiles instead of 3 of 216, 1.07x; M = 1024).
PairShape pair_shape(bool sparse, int M, int N) {
  return pair_shape_for(sparse, M, N, sm_count() / 2 > 0 ? sm_count() / 2 : 1);
}

PairShape pair_shape_for(bool sparse, int M, int N, int64_t clusters) {
  if (clusters < 1) clusters = 1;
  auto cost = [&](int rb, int tn, double bytes_per_kmac) {
    const int64_t tiles = ((M + 256 * rb - 1) / (256 * rb)) * static_cast<int64_t>((N + tn - 1) / tn);
    const int64_t waves = (tiles + clusters - 1) / clusters;
    return static_cast<double>(waves) * 256.0 * rb * tn * bytes_per_kmac;
  };
  if (!sparse) return cost(1, 448, 0.965) < cost(1, 256, 1.0) ? PairShape{1, 448} : PairShape{1, 256};
  const PairShape cand[4] = {{2, 224}, {2, 192}, {1, 256}, {1, 192}};
  const double bytes[4] = {21.3, 22.9, 23.8, 26.7};
  int best = 0;
  double best_cost = cost(cand[0].rb, cand[0].tn, bytes[0]);
  for (int i = 1; i < 4; ++i) {
    const double c = cost(cand[i].rb, cand[i].tn, bytes[i]);
    if (c < best_cost) {
      best = i;
      best_cost = c;
    }
  }
  return cand[best];
}

bool pair_shape_valid(bool sparse, PairShape shape) {
  if (!sparse) return shape.rb == 1 && (shape.tn == 256 || shape.tn == 448);
  return (shape.rb == 2 && (shape.tn == 224 || shape.tn == 192)) || (shape.rb == 1 && (shape.tn == 256 || shape.tn == 192));
}

int gelu_norm_slots(bool sparse, PairShape shape, int N) {
  const int cols = shape.rb == 2 ? shape.tn : shape.tn / 2;  // columns of one epilogue warp
  (void)sparse;
  return ((N + shape.tn - 1) / shape.tn) * (shape.tn / cols);
}

}  // namespace lynx
