/* A plain C99 program against include/kda.h: the header compiles as C, the
 * library links, and its host-side entry points answer without a GPU.  Every
 * kda_fwd / kda_bwd call below is built to fail host validation, which comes
 * before any launch, so the fake pointers are never dereferenced. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "kda.h"

#define FAKE ((void*)(uintptr_t)(1u << 20)) /* non-null, 256-byte aligned */

static int fails = 0;

static void expect(const char* what, long got, long want) {
  if (got != want) {
    printf("FAIL %s: got %ld, want %ld\n", what, got, want);
    fails++;
  }
}

static kda_problem problem(int dk, int dv) {
  kda_problem p;
  memset(&p, 0, sizeof p);
  p.B = 2;
  p.T = 256;
  p.H = 4;
  p.dk = dk;
  p.dv = dv;
  p.dtype = KDA_BF16;
  p.scale = 0.f;
  p.gate = KDA_GATE_CHANNEL;
  return p;
}

static kda_status fwd(const kda_problem* p, void* q, void* ws, size_t ws_bytes) {
  return kda_fwd(p, q, FAKE, FAKE, FAKE, FAKE, (const float*)FAKE, (const float*)FAKE, NULL, FAKE, NULL, 1, ws,
                 ws_bytes, (cudaStream_t)0);
}

static kda_status bwd(const kda_problem* p, void* ws, size_t ws_bytes) {
  return kda_bwd(p, FAKE, FAKE, FAKE, FAKE, FAKE, (const float*)FAKE, (const float*)FAKE, NULL, FAKE, NULL, FAKE,
                 FAKE, FAKE, FAKE, FAKE, (float*)FAKE, (float*)FAKE, NULL, ws, ws_bytes, (cudaStream_t)0);
}

int main(void) {
  kda_problem p = problem(32, 64), bad = problem(48, 64), none = problem(32, 64);
  none.H = 0;
  const size_t ws_f = kda_workspace_size(&p, 0), ws_b = kda_workspace_size(&p, 1);
  expect("forward workspace is sized", ws_f > 0, 1);
  expect("the backward's workspace holds the forward's", ws_b >= ws_f, 1);
  expect("no workspace for an invalid problem", (long)kda_workspace_size(&none, 1), 0);
  expect("unsupported head shape", fwd(&bad, FAKE, FAKE, ws_b), KDA_ERR_UNSUPPORTED);
  expect("null input", fwd(&p, NULL, FAKE, ws_b), KDA_ERR_INVALID_ARG);
  expect("misaligned input", fwd(&p, (char*)FAKE + 2, FAKE, ws_b), KDA_ERR_ALIGNMENT);
  expect("missing workspace", fwd(&p, FAKE, NULL, 0), KDA_ERR_WORKSPACE);
  expect("workspace too small", fwd(&p, FAKE, FAKE, ws_f - 1), KDA_ERR_WORKSPACE);
  expect("backward, workspace too small", bwd(&p, FAKE, 16), KDA_ERR_WORKSPACE);
  expect("backward, unsupported head shape", bwd(&bad, FAKE, ws_b), KDA_ERR_UNSUPPORTED);
  const char* ok = kda_strerror(KDA_OK);
  const char* ws = kda_strerror(KDA_ERR_WORKSPACE);
  expect("status texts", ok != NULL && ws != NULL && strlen(ws) > 0 && strcmp(ok, ws) != 0, 1);
  printf(fails ? "FAILED (%d)\n" : "ok\n", fails);
  return fails != 0;
}
