"""GB300-native W4A8 GEMM (QoQ / QServe hot path)."""
