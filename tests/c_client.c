/* A plain C client of libcredit.so: includes only include/credit.h, links the
 * library, and calls entry points whose answers need no GPU (argument
 * rejection, status strings, the build kind, the version). */
#include <stdio.h>
#include <string.h>

#include "credit.h"

int main(void) {
    int bad = 0;
    credit_plan_t req, out;
    memset(&req, 0, sizeof(req));
    if (credit_plan(CREDIT_SOFTMAX, 4, 4, CREDIT_F32, 0, NULL) != CREDIT_ERR_INVALID_ARG) bad |= 1;
    if (credit_softmax(NULL, NULL, 4, 4, CREDIT_F32, NULL, NULL, 0, NULL) != CREDIT_ERR_INVALID_ARG)
        bad |= 2;
    req.variant = CREDIT_TWO_PASS;
    req.exchange = CREDIT_EXCHANGE_ASYNC;  /* no exchange in a two-pass plan */
    if (credit_plan_with(CREDIT_LAYERNORM, 4, 4, CREDIT_BF16, 0, &req, &out) != CREDIT_ERR_INVALID_ARG)
        bad |= 4;
    if (strcmp(credit_status_string(CREDIT_OK), "ok") != 0) bad |= 8;
    if (credit_debug_build() != 0) bad |= 16;
    printf("%s %d\n", credit_version(), bad);
    return bad;
}
