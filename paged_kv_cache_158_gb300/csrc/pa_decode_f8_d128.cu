#define PA_D 128
#define PA_F8 1
#include "pa_decode_inst.inc"
