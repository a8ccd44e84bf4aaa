/* Prints the sizes and field offsets of the C ABI's structures (include/dflash2.h),
 * one "name value" per line, for the binding's layout test. */
#include <stddef.h>
#include <stdio.h>

#include "dflash2.h"

#define OFF(T, f) printf(#T "." #f " %zu\n", offsetof(T, f))

int main(void) {
  printf("dflash2_config %zu\n", sizeof(dflash2_config));
  OFF(dflash2_config, hidden);
  OFF(dflash2_config, mask_token_id);
  OFF(dflash2_config, weight_format);
  OFF(dflash2_config, rope_theta);
  OFF(dflash2_config, rms_eps);
  printf("dflash2_matrix %zu\n", sizeof(dflash2_matrix));
  printf("dflash2_layer_weights %zu\n", sizeof(dflash2_layer_weights));
  OFF(dflash2_layer_weights, mlp_base);
  OFF(dflash2_layer_weights, q);
  OFF(dflash2_layer_weights, mlp_delta);
  printf("dflash2_weights %zu\n", sizeof(dflash2_weights));
  OFF(dflash2_weights, final_norm);
  OFF(dflash2_weights, fc);
  OFF(dflash2_weights, cb_b);
  OFF(dflash2_weights, layers);
  printf("dflash2_step_args %zu\n", sizeof(dflash2_step_args));
  OFF(dflash2_step_args, anchor_ids);
  OFF(dflash2_step_args, status);
  OFF(dflash2_step_args, width);
  return 0;
}
