// Host-side harness: runs the library's correctly rounded fp32 power
// (double-double exp/log, the arithmetic of the smoothing-factor kernel)
// on the CPU.  Reads lines "xbits ybits" (hex fp32 bit patterns) on stdin
// and prints the result's bit pattern for each.
#include <stdio.h>

#include "smooth.cu"

int main() {
  unsigned xb, yb;
  while (scanf("%x %x", &xb, &yb) == 2) {
    float x, y;
    memcpy(&x, &xb, 4);
    memcpy(&y, &yb, 4);
    float r = sq::pow_cr(x, y);
    unsigned rb;
    memcpy(&rb, &r, 4);
    printf("%08x\n", rb);
  }
  return 0;
}
