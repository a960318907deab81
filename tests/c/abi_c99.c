/* Plain C99 user of the C ABI (include/fp8bs.h): it compiles without any
 * CUDA header, links against libfp8bs.so and calls entry points that need
 * no GPU.  Built and run by tests/test_abi_cpu.py. */
#include <stdio.h>
#include <string.h>

#include "fp8bs.h"

int main(void) {
    int bad = 0;
    if (fp8bs_version() < 102) { printf("version %d\n", fp8bs_version()); ++bad; }
    if (fp8bs_workspace_size() != FP8BS_WORKSPACE_BYTES) { printf("workspace size\n"); ++bad; }
    if (fp8bs_workspace_size_for(FP8BS_OP_QUANTIZE, 4, 128, FP8BS_TOKEN_1x128, 0) != 0) {
        printf("workspace for 1x128\n");
        ++bad;
    }
    if (strlen(fp8bs_status_string(FP8BS_EINVAL)) == 0) { printf("status string\n"); ++bad; }
    /* Host-side argument checks return before anything touches the device. */
    char fake[64];
    if (fp8_quantize(NULL, 4, 128, 128, FP8BS_TOKEN_1x128, fake, fake, NULL, 0u, NULL, 0, NULL) != FP8BS_EINVAL) {
        printf("null input accepted\n");
        ++bad;
    }
    if (fp8_block_gemm(fake, fake, FP8BS_TOKEN_1x128, fake, fake, FP8BS_BLOCK_128x128, NULL, NULL, 128, 128, 256,
                       fake, 7, fake, FP8BS_WORKSPACE_BYTES, NULL) != FP8BS_EINVAL) {
        printf("unknown output type accepted\n");
        ++bad;
    }
    if (fp8_block_gemm(fake, fake, FP8BS_TOKEN_1x128, fake, fake, FP8BS_BLOCK_128x128, NULL, NULL, 128, 132, 256,
                       fake, FP8BS_OUT_F32, fake, FP8BS_WORKSPACE_BYTES, NULL) != FP8BS_EINVAL) {
        printf("n %% 8 != 0 accepted\n");
        ++bad;
    }
    if (bad == 0) printf("c99 abi ok\n");
    return bad;
}
