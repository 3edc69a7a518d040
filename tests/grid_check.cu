// Host harness for the grid-order and tile-range helpers of the kernels
// (compiled and run by test_grid_host.py; no device code runs).
#include <cstdio>
#include <cstdlib>
#include "../io_aware_exact_10_gb300/csrc/fa_kernels.h"

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  const char* what = argv[1];
  if (what[0] == 'd') {  // decode_grid BH tiles group -> one "bh rank" line per L
    const int BH = atoi(argv[2]), tiles = atoi(argv[3]), group = atoi(argv[4]);
    for (int L = 0; L < BH * tiles; ++L) {
      const fa::GridPos p = fa::decode_grid(L, BH, tiles, group);
      printf("%d %d\n", p.bh, p.rank);
    }
  } else if (what[0] == 'f') {  // first_query_tile nkv coff -> one value per key tile
    const int nkv = atoi(argv[2]), coff = atoi(argv[3]);
    for (int kt = 0; kt < nkv; ++kt) printf("%d\n", fa::first_query_tile(kt, coff));
  } else if (what[0] == 'h') {  // head_group BH tiles sms
    printf("%d\n", fa::head_group(atoi(argv[2]), atoi(argv[3]), atoi(argv[4])));
  } else if (what[0] == 'p') {  // persistent_launch causal sparse tiles
    printf("%d\n", (int)fa::persistent_launch(atoi(argv[2]) != 0, atoi(argv[3]) != 0, atoi(argv[4])));
  } else if (what[0] == 'u') {  // decode_pair BH tiles -> one "bh rank" line per L
    const int BH = atoi(argv[2]), tiles = atoi(argv[3]);
    for (int L = 0; L < BH * tiles; ++L) {
      const fa::GridPos p = fa::decode_pair(L, tiles);
      printf("%d %d\n", p.bh, p.rank);
    }
  } else if (what[0] == 'l') {  // pair_launch causal sparse square tiles items sms max_tiles
    printf("%d\n", (int)fa::pair_launch(atoi(argv[2]) != 0, atoi(argv[3]) != 0, atoi(argv[4]) != 0,
                                       atoi(argv[5]), atol(argv[6]), atoi(argv[7]), atoi(argv[8])));
  }
  return 0;
}
