#define PA_D 64
#define PA_F8 0
#include "pa_decode_inst.inc"
