/* Prints Philox4x32-10 output blocks from the cuRAND host generator (a library
 * implementation of the same generator), used to pin the oracle's Philox.
 * Usage: curand_philox_blocks <seed> <first_block> <n_blocks>
 * Output block b (4 words) is printed in generation order; the test maps b to
 * the generator's counter and compares under key (seed lo32, seed hi32). */
#include <stdio.h>
#include <stdlib.h>
#include <curand.h>

int main(int argc, char** argv) {
  if (argc != 4) return 2;
  unsigned long long seed = strtoull(argv[1], NULL, 0);
  unsigned long long first = strtoull(argv[2], NULL, 0);
  size_t n = (size_t)strtoull(argv[3], NULL, 0);
  curandGenerator_t g;
  if (curandCreateGeneratorHost(&g, CURAND_RNG_PSEUDO_PHILOX4_32_10) != CURAND_STATUS_SUCCESS) return 3;
  if (curandSetPseudoRandomGeneratorSeed(g, seed) != CURAND_STATUS_SUCCESS) return 3;
  if (curandSetGeneratorOffset(g, 4ULL * first) != CURAND_STATUS_SUCCESS) return 3;
  unsigned int* out = (unsigned int*)malloc(4 * n * sizeof(unsigned int));
  if (curandGenerate(g, out, 4 * n) != CURAND_STATUS_SUCCESS) return 3;
  for (size_t i = 0; i < 4 * n; i++) printf("%u\n", out[i]);
  free(out);
  curandDestroyGenerator(g);
  return 0;
}
