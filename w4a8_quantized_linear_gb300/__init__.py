"""GB300-native W8A8 / W4A8 online-activation-quantized linear layer."""
