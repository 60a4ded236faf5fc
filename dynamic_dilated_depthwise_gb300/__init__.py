"""GB300-native DDPM core: fused generator + dynamic dilated depthwise filter."""
