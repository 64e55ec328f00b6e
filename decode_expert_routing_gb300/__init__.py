"""GB300-native MoE decode routing: router GEMV, top-k gate, sort, MXFP8 quant."""
